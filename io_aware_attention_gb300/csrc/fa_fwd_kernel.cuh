// Attention forward for sm_103a: tcgen05 tensor cores + TMEM + TMA.
//
// One CTA owns BM = 128 query rows of one (batch, head) and streams the key /
// value rows in tiles of BN = 128 through shared memory, carrying the
// online-softmax state per row ("Kernels — fusion and FlashAttention" §3–§4;
// "Fusion and IO-aware kernels" § FlashAttention, steps 1–4):
//
//   S_j   = Q K_j^T                        (tcgen05.mma, smem x smem -> TMEM fp32)
//   m_new = max(m, rowmax(S_j) * c)        (c = scale * log2 e, base-2 units)
//   P_j   = 2^(S_j * c - m)                (bf16, written into TMEM)
//   l     = l * 2^(m_old - m_new) + rowsum(P_j)              (fp32 values)
//   [O|l~]= [O|l~] * 2^(m_old - m_new) + P_j [V_j | 1]       (tcgen05.mma, TMEM x smem)
//   out   = O / l~,   lse = (m + log2 l) * ln 2
//
// The score matrix lives only in TMEM, one 128x128 tile at a time.
//
// Warp roles (320 threads):
//   warps 0-7  softmax.  Warp w serves query rows 32*(w%4) .. +31 (its TMEM
//              lane quarter) and score columns 64*(w/4) .. +63, so every SM
//              sub-partition runs two softmax warps.  Each thread owns half a
//              row: masking, partial row max (exchanged with the partner half
//              through shared memory), exponentials, its half of P, and its
//              half of the O columns for rescaling and the epilogue.
//   warp 8     TMA producer: Q once, then K_j / V_j into rings of stages.
//   warp 9     MMA issuer (one thread), also allocates TMEM.
//
// TMEM columns (512 allocated, lanes = query rows):
//   [  0,128) S buffer 0     [128,256) S buffer 1   (fp32 scores, double-buffered)
//   [256,256+d) O (fp32)     [256+d, 256+d+16) l~ (16 equal copies)
//   [TM_P, TM_P+64) P (bf16 pairs)
// S_{j+1} is computed while the softmax works on S_j.  P has its own columns,
// so no MMA ever overwrites TMEM that an earlier, still-running MMA reads.
//
// l~ = rowsum(bf16(P)): each V stage carries a 64-wide block of ones after
// its d value columns, and the P.V MMA runs with N = d + 16, so the tensor
// core sums exactly the rounded probabilities it multiplies.  O / l~ is then
// an exact convex combination of the value rows even though P is rounded.
//
// Rescaling is lazy: a row keeps its reference max until a tile raises the
// max by more than RESCALE_LOG2 (base-2 units); P, l and l~ share the same
// reference, so the ratios are unaffected and P stays below 2^RESCALE_LOG2.
//
// Every wait is bounded in time; on expiry the thread records the wait in the
// device status word, raises a CTA-wide abort flag, and all roles drain their
// in-flight copies / MMAs and reach the common exit, where TMEM is freed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fa {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // keys per K/V tile
constexpr int SOFTMAX_THREADS = 256;
constexpr int NUM_THREADS = SOFTMAX_THREADS + 64;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256;
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t BLK_BYTES = BN * 128;  // one 64-column, 128-row swizzled block (16 KB)

constexpr uint32_t STATUS_TIMEOUT = 1u;

// Named barriers (0 is __syncthreads).
constexpr uint32_t NB_SOFTMAX = 1;

struct Params {
    float* lse;
    int N;
    int num_m_blocks;
    float scale_log2;  // scale * log2(e)
    unsigned long long wait_limit_ns;
};

template <int D>
struct Layout {
    static_assert(D == 64 || D == 128, "head size");
    static constexpr int STAGES = (D == 128) ? 2 : 4;
    static constexpr int DBLK = D / 64;                   // 64-column blocks of a row
    static constexpr uint32_t TM_L = TM_O + D;            // l~ columns
    static constexpr uint32_t TM_P = (D == 128) ? 448 : 384;
    static_assert(TM_L + 16 <= TM_P && TM_P + 64 <= TM_COLS, "TMEM budget");
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;      // bytes of one K or V tile
    static constexpr uint32_t VSTAGE = (DBLK + 1) * BLK_BYTES;  // V blocks + the ones block
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
    static constexpr uint32_t OFF_RED = OFF_V + STAGES * VSTAGE;  // float[2][2][BM] + float[2][BM]
    static constexpr uint32_t RED_BYTES = 6 * BM * 4;
    static constexpr uint32_t OFF_BAR = OFF_RED + RED_BYTES;
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + STAGES;
    static constexpr int B_VFULL = B_KEMPTY + STAGES;
    static constexpr int B_VEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_VEMPTY + STAGES;  // 2
    static constexpr int B_PFULL = B_SFULL + 2;
    static constexpr int B_ODONE = B_PFULL + 1;
    static constexpr int B_DRAIN = B_ODONE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort
    static constexpr uint32_t USED = OFF_MISC + 16;
    static constexpr uint32_t SMEM_BYTES = USED + 1024;  // + slack to align the base to 1024
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ unsigned int g_status;        // STATUS_* bits, sticky until read by the host
__device__ unsigned int g_status_where;  // first wait code that gave up (+1)

__device__ __forceinline__ void record_timeout(uint32_t code, volatile uint32_t* abort_flag)
{
    *abort_flag = 1u;
    atomicCAS(&g_status_where, 0u, code + 1u);
    atomicOr(&g_status, STATUS_TIMEOUT);
}

// Bounded wait on an mbarrier phase.  Gives up (returns false) when the CTA
// has aborted or after `limit_ns`, in which case it raises the abort.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                         volatile uint32_t* abort_flag, uint32_t code)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) {
            record_timeout(code, abort_flag);
            return false;
        }
    }
}

// Bounded wait used while draining: ignores the abort flag (in-flight copies
// must land before the CTA exits) but still gives up after `limit_ns`.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile uint32_t* abort_flag, uint32_t code)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > limit_ns) {
            record_timeout(code, abort_flag);
            return;
        }
    }
}

// All 32 lanes wait; the result is made warp-uniform.
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                              volatile uint32_t* abort_flag, uint32_t code)
{
    const bool ok = wait_bar(bar, parity, limit_ns, abort_flag, code);
    return __all_sync(0xffffffffu, ok);
}

// Max of 64 values with 3-input max instructions (depth 4).
__device__ __forceinline__ float max64(const float (&s)[64])
{
    float t[22];
#pragma unroll
    for (int i = 0; i < 21; ++i) t[i] = ptx::fmax3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
    t[21] = s[63];
    float u[8];
#pragma unroll
    for (int i = 0; i < 7; ++i) u[i] = ptx::fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[7] = t[21];
    return ptx::fmax3(ptx::fmax3(u[0], u[1], u[2]), ptx::fmax3(u[3], u[4], u[5]), fmaxf(u[6], u[7]));
}

// Multiplies this thread's D/2 O columns (TMEM, from `taddr`) by `corr`.
template <int D>
__device__ __forceinline__ void scale_cols(uint32_t taddr, float corr)
{
    const uint64_t c2 = ptx::f2_pack(corr, corr);
#pragma unroll
    for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t o[32];
        ptx::tmem_ld32(taddr + ch * 32, o);
        ptx::tmem_wait_ld(o);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            uint64_t x = ptx::f2_pack(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1]));
            x = ptx::f2_mul(x, c2);
            float a, b;
            ptx::f2_unpack(x, a, b);
            o[2 * c] = __float_as_uint(a);
            o[2 * c + 1] = __float_as_uint(b);
        }
        ptx::tmem_st32(taddr + ch * 32, o);
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const Params p)
{
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* const sgen = smem_raw + (sbase - raw);
    volatile uint32_t* const misc = reinterpret_cast<volatile uint32_t*>(sgen + L::OFF_MISC);
    volatile uint32_t* const abort_flag = misc + 1;
    float* const red = reinterpret_cast<float*>(sgen + L::OFF_RED);  // [2 slots][2 halves][BM]
    float* const red_l = red + 4 * BM;                               // [2 halves][BM]
    auto bar = [&](int i) -> uint32_t { return sbase + L::OFF_BAR + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;

    // Work item: heaviest query blocks of a head first (causal rows near the
    // end see the most keys); the blocks of one head run side by side so its
    // K/V stay in L2.
    const int m_block = p.num_m_blocks - 1 - (int)(blockIdx.x % (unsigned)p.num_m_blocks);
    const int bh = (int)(blockIdx.x / (unsigned)p.num_m_blocks);
    const int q0 = m_block * BM;
    const int N = p.N;
    const int n_kv_all = (N + BN - 1) / BN;
    const int n_kv = CAUSAL ? min(n_kv_all, (q0 + BM - 1) / BN + 1) : n_kv_all;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(L::B_Q), 1);
        for (int s = 0; s < L::STAGES; ++s) {
            ptx::mbar_init(bar(L::B_KFULL + s), 1);
            ptx::mbar_init(bar(L::B_KEMPTY + s), 1);
            ptx::mbar_init(bar(L::B_VFULL + s), 1);
            ptx::mbar_init(bar(L::B_VEMPTY + s), 1);
        }
        ptx::mbar_init(bar(L::B_SFULL + 0), 1);
        ptx::mbar_init(bar(L::B_SFULL + 1), 1);
        ptx::mbar_init(bar(L::B_PFULL), SOFTMAX_THREADS);
        ptx::mbar_init(bar(L::B_ODONE), 1);
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp < 8) {
        // The ones block of every V stage: bf16 1.0 everywhere (any swizzle).
        const uint32_t one2 = 0x3F803F80u;
        for (int s = 0; s < L::STAGES; ++s) {
            const uint32_t blk = sbase + L::OFF_V + s * L::VSTAGE + L::DBLK * BLK_BYTES;
#pragma unroll
            for (int i = 0; i < (int)(BLK_BYTES / 16 / SOFTMAX_THREADS); ++i)
                ptx::st_shared_v4(blk + 16u * (threadIdx.x + i * SOFTMAX_THREADS), one2, one2, one2, one2);
        }
        ptx::fence_proxy_async_smem();
    }
    if (warp == WARP_TMA && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
    }
    if (warp == WARP_MMA) {
        ptx::tmem_alloc(sbase + L::OFF_MISC, TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    if (warp == WARP_TMA) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(L::B_Q), L::Q_BYTES);
            for (int c = 0; c < L::DBLK; ++c)
                ptx::tma_load_3d(sbase + L::OFF_Q + c * BLK_BYTES, &tm_q, bar(L::B_Q), c * 64, q0, bh);
            int nk = 0, nv = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % L::STAGES;
                const uint32_t ph = (uint32_t)(j / L::STAGES) & 1u;
                if (!wait_bar(bar(L::B_KEMPTY + s), ph ^ 1u, limit, abort_flag, 0x100 + L::B_KEMPTY + s)) break;
                ptx::mbar_arrive_expect_tx(bar(L::B_KFULL + s), L::KV_BYTES);
                for (int c = 0; c < L::DBLK; ++c)
                    ptx::tma_load_3d(sbase + L::OFF_K + s * L::KV_BYTES + c * BLK_BYTES, &tm_k,
                                     bar(L::B_KFULL + s), c * 64, j * BN, bh);
                ++nk;
                if (!wait_bar(bar(L::B_VEMPTY + s), ph ^ 1u, limit, abort_flag, 0x100 + L::B_VEMPTY + s)) break;
                ptx::mbar_arrive_expect_tx(bar(L::B_VFULL + s), L::KV_BYTES);
                for (int c = 0; c < L::DBLK; ++c)
                    ptx::tma_load_3d(sbase + L::OFF_V + s * L::VSTAGE + c * BLK_BYTES, &tm_v,
                                     bar(L::B_VFULL + s), c * 64, j * BN, bh);
                ++nv;
            }
            // Drain: every copy this thread issued must land before exit.
            drain_bar(bar(L::B_Q), 0, limit, abort_flag, 0x180);
            for (int j = max(0, nk - L::STAGES); j < nk; ++j)
                drain_bar(bar(L::B_KFULL + j % L::STAGES), (uint32_t)(j / L::STAGES) & 1u, limit,
                          abort_flag, 0x181);
            for (int j = max(0, nv - L::STAGES); j < nv; ++j)
                drain_bar(bar(L::B_VFULL + j % L::STAGES), (uint32_t)(j / L::STAGES) & 1u, limit,
                          abort_flag, 0x182);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(BM, D + 16, true);
            bool ok = wait_bar(bar(L::B_Q), 0, limit, abort_flag, 0x200 + L::B_Q);
            // S_j = Q K_j^T into S buffer (j & 1); K-major operands, 16 columns per MMA.
            auto issue_s = [&](int j) -> bool {
                const int s = j % L::STAGES;
                if (!wait_bar(bar(L::B_KFULL + s), (uint32_t)(j / L::STAGES) & 1u, limit, abort_flag,
                              0x200 + L::B_KFULL + s))
                    return false;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem + ((j & 1) ? TM_S1 : TM_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (uint32_t)(kk >> 2) * BLK_BYTES + (uint32_t)(kk & 3) * 32;
                    const uint64_t a = ptx::sdesc_sw128(sbase + L::OFF_Q + koff, 16, 1024);
                    const uint64_t b = ptx::sdesc_sw128(sbase + L::OFF_K + s * L::KV_BYTES + koff, 16, 1024);
                    ptx::mma_ss(d_tmem, a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(bar(L::B_KEMPTY + s));
                ptx::tc_commit(bar(L::B_SFULL + (j & 1)));
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n_kv > 1) ok = issue_s(1);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j % L::STAGES;
                if (!wait_bar(bar(L::B_PFULL), (uint32_t)j & 1u, limit, abort_flag, 0x200 + L::B_PFULL))
                    break;
                if (!wait_bar(bar(L::B_VFULL + s), (uint32_t)(j / L::STAGES) & 1u, limit, abort_flag,
                              0x200 + L::B_VFULL + s))
                    break;
                ptx::tc_fence_after_sync();
                // [O | l~] (+)= P_j [V_j | 1]: A = P from TMEM (2 bf16 per column,
                // 8 columns per 16 keys); B MN-major (value columns contiguous):
                // 64-column blocks BLK_BYTES apart (the ones block follows the
                // value blocks), 8-key groups 1024 bytes apart.
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bdesc = ptx::sdesc_sw128(
                        sbase + L::OFF_V + s * L::VSTAGE + (uint32_t)kk * (16 * 128), BLK_BYTES, 1024);
                    ptx::mma_ts(tmem + TM_O, tmem + L::TM_P + (uint32_t)kk * 8, bdesc, IDESC_O,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::tc_commit(bar(L::B_VEMPTY + s));
                ptx::tc_commit(bar(L::B_ODONE));
                if (j + 2 < n_kv) ok = issue_s(j + 2);
            }
            // Drain: all MMAs issued by this thread complete before TMEM is freed.
            ptx::tc_commit(bar(L::B_DRAIN));
            drain_bar(bar(L::B_DRAIN), 0, limit, abort_flag, 0x280);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax warps
        const int quarter = warp & 3;
        const int half = warp >> 2;               // score columns [64*half, 64*half+64)
        const int row = quarter * 32 + lane;      // query row in the tile == TMEM lane
        const int q_idx = q0 + row;
        const int key_max = CAUSAL ? min(q_idx, N - 1) : N - 1;
        const int cta_key_max = CAUSAL ? min(q0, N - 1) : N - 1;  // smallest key_max of the CTA
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t o_cols = tmem + lane_off + TM_O + (uint32_t)half * (D / 2);
        const uint32_t l_cols = tmem + lane_off + L::TM_L + (uint32_t)half * 8;
        const float sl2 = p.scale_log2;
        const uint64_t sl2_2 = ptx::f2_pack(sl2, sl2);
        float m_ref = -INFINITY;
        uint64_t lacc[4] = {0, 0, 0, 0};  // fp32 pairs: this half-row's sum of probabilities
        bool ok = true;

        // Every softmax warp runs all n_kv iterations and reaches each named
        // barrier the same number of times, also after an abort (ok == false:
        // the work is skipped, the barriers are not), so a named barrier can
        // never wait for a warp that has left the loop.
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            if (ok) {
                ok = warp_wait_bar(bar(L::B_SFULL + b), (uint32_t)(j >> 1) & 1u, limit, abort_flag,
                                   0x300 + L::B_SFULL + b);
            }
            float s[64];
            float mx = -INFINITY;
            if (ok) {
                ptx::tc_fence_after_sync();
                uint32_t r0[32], r1[32];
                const uint32_t s_tmem = tmem + lane_off + (b ? TM_S1 : TM_S0) + (uint32_t)half * 64;
                ptx::tmem_ld32(s_tmem + 0, r0);
                ptx::tmem_ld32(s_tmem + 32, r1);
                ptx::tmem_wait_ld(r0);
                ptx::reg_fence(r1);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    s[c] = __uint_as_float(r0[c]);
                    s[32 + c] = __uint_as_float(r1[c]);
                }
                // Causal diagonal tile / keys past N: -inf before the max.
                const int k0 = j * BN + half * 64;
                if (j * BN + BN - 1 > cta_key_max) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (k0 + c > key_max) s[c] = -INFINITY;
                }
                mx = max64(s);
                red[(b * 2 + half) * BM + row] = mx;
            }
            // Row max: this half's, then the partner half's through shared memory.
            ptx::named_barrier_sync(NB_SOFTMAX, SOFTMAX_THREADS);
            if (!ok) continue;
            mx = fmaxf(mx, red[(b * 2 + (half ^ 1)) * BM + row]);
            const float m_tile = mx * sl2;  // scale > 0, so max commutes with it

            bool waited = false;
            if (j == 0) {
                m_ref = (m_tile == -INFINITY) ? 0.f : m_tile;
            } else {
                const float m_new = fmaxf(m_ref, m_tile);
                const bool need = m_new > m_ref + RESCALE_LOG2;
                // Both halves of a row see the same values, so they decide alike.
                if (__any_sync(0xffffffffu, need)) {
                    // [O | l~] hold P_{j-1} [V_{j-1} | 1] once that MMA is done.
                    ok = warp_wait_bar(bar(L::B_ODONE), (uint32_t)(j - 1) & 1u, limit, abort_flag,
                                       0x300 + L::B_ODONE);
                    if (!ok) continue;
                    waited = true;
                    ptx::tc_fence_after_sync();
                    const float corr = ptx::ex2(m_ref - m_new);
                    const uint64_t c2 = ptx::f2_pack(corr, corr);
#pragma unroll
                    for (int i = 0; i < 4; ++i) lacc[i] = ptx::f2_mul(lacc[i], c2);
                    m_ref = m_new;
                    scale_cols<D>(o_cols, corr);
                    uint32_t lt[8];
                    ptx::tmem_ld8(l_cols, lt);
                    ptx::tmem_wait_ld_only();
                    ptx::reg_fence8(lt);
#pragma unroll
                    for (int c = 0; c < 8; ++c) lt[c] = __float_as_uint(__uint_as_float(lt[c]) * corr);
                    ptx::tmem_st8(l_cols, lt);
                    ptx::tmem_wait_st();
                }
            }

            // P = 2^(s*c - m_ref), two lanes of fp32 per instruction; rounded to
            // bf16 for the P.V MMA.
            const uint64_t negm2 = ptx::f2_pack(-m_ref, -m_ref);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const uint64_t x = ptx::f2_fma(ptx::f2_pack(s[2 * c], s[2 * c + 1]), sl2_2, negm2);
                float x0, x1;
                ptx::f2_unpack(x, x0, x1);
                const float a0 = ptx::ex2(x0), a1 = ptx::ex2(x1);
                lacc[c & 3] = ptx::f2_add(lacc[c & 3], ptx::f2_pack(a0, a1));
                pk[c] = ptx::pack_bf16x2(a0, a1);
            }

            // The single P buffer was last read by the MMA of tile j-1.
            if (j >= 1 && !waited) {
                ok = warp_wait_bar(bar(L::B_ODONE), (uint32_t)(j - 1) & 1u, limit, abort_flag,
                                   0x340 + L::B_ODONE);
                if (!ok) continue;
                ptx::tc_fence_after_sync();
            }
            ptx::tmem_st32(tmem + lane_off + L::TM_P + (uint32_t)half * 32, pk);
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(L::B_PFULL));
        }

        // ------------------------------------------------------- epilogue
        if (ok) ok = warp_wait_bar(bar(L::B_ODONE), (uint32_t)(n_kv - 1) & 1u, limit, abort_flag,
                                   0x380 + L::B_ODONE);
        float l_half;
        {
            float a, c;
            const uint64_t t = ptx::f2_add(ptx::f2_add(lacc[0], lacc[1]), ptx::f2_add(lacc[2], lacc[3]));
            ptx::f2_unpack(t, a, c);
            l_half = a + c;
        }
        red_l[half * BM + row] = l_half;
        ptx::named_barrier_sync(NB_SOFTMAX, SOFTMAX_THREADS);
        if (ok) {
            ptx::tc_fence_after_sync();
            const float l = l_half + red_l[(half ^ 1) * BM + row];
            uint32_t lt[8];
            ptx::tmem_ld8(l_cols, lt);
            ptx::tmem_wait_ld_only();
            ptx::reg_fence8(lt);
            const float inv_l = 1.0f / __uint_as_float(lt[0]);
            // O half-row -> bf16 -> the Q tile's shared memory (Q is no longer
            // read), in the 128-byte-swizzled layout the O tensor map expects.
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) {
                uint32_t o[32];
                ptx::tmem_ld32(o_cols + ch * 32, o);
                ptx::tmem_wait_ld(o);
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    w[c] = ptx::pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                            __uint_as_float(o[2 * c + 1]) * inv_l);
                const int col0 = half * (D / 2) + ch * 32;
                const uint32_t blk = sbase + L::OFF_Q + (uint32_t)(col0 >> 6) * BLK_BYTES + (uint32_t)row * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t chunk = (uint32_t)(((col0 & 63) >> 3) + u);
                    ptx::st_shared_v4(blk + ((chunk ^ (uint32_t)(row & 7)) << 4), w[4 * u], w[4 * u + 1],
                                      w[4 * u + 2], w[4 * u + 3]);
                }
            }
            if (half == 0 && q_idx < N)
                p.lse[(int64_t)bh * N + q_idx] = (m_ref + ptx::lg2(l)) * 0.69314718055994530942f;
        }
        ptx::fence_proxy_async_smem();
        ptx::named_barrier_sync(NB_SOFTMAX, SOFTMAX_THREADS);
        if (threadIdx.x == 0 && *abort_flag == 0u) {
            for (int c = 0; c < L::DBLK; ++c)
                ptx::tma_store_3d(&tm_o, sbase + L::OFF_Q + c * BLK_BYTES, c * 64, q0, bh);
            ptx::tma_store_commit();
            ptx::tma_store_wait_read();
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace fa
