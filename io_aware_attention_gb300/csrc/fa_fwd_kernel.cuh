// Attention forward for sm_103a: tcgen05 tensor cores + TMEM + TMA.
//
// One CTA owns BM = 128 query rows of one (batch, head) and streams the key /
// value rows in tiles of BN = 128 through shared memory, carrying the
// online-softmax state per row ("Kernels — fusion and FlashAttention" §3–§4;
// "Fusion and IO-aware kernels" § FlashAttention, steps 1–4):
//
//   S_j   = Q K_j^T                        (tcgen05.mma, smem x smem -> TMEM fp32)
//   m_new = max(m, rowmax(S_j) * c)        (c = scale * log2 e, base-2 units)
//   P_j   = 2^(S_j * c - m)                (bf16, written back into TMEM)
//   l     = l * 2^(m_old - m_new) + rowsum(P_j)          (fp32 values)
//   l~    = l~ * 2^(m_old - m_new) + rowsum(bf16(P_j))   (the values the MMA sees)
//   O     = O * 2^(m_old - m_new) + P_j V_j (tcgen05.mma, TMEM x smem -> TMEM fp32)
//   out   = O / l~,   lse = (m + log2 l) * ln 2
//
// The score matrix lives only in TMEM, one 128x128 tile at a time.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t); masking,
//              row max, exponentials, P store, O rescale, epilogue.
//   warp 4     TMA producer: Q once, then K_j / V_j into a ring of stages.
//   warp 5     MMA issuer (one thread), also allocates TMEM.
//
// TMEM columns (512 allocated, lanes = query rows):
//   [  0,128) S buffer 0     [128,256) S buffer 1   (fp32 scores, double-buffered)
//   [256,256+d) O accumulator (fp32)
//   [384,448) P buffer 0     [448,512) P buffer 1   (bf16 pairs)
// S_{j+1} is computed while the softmax works on S_j.  P has its own buffers,
// so no MMA ever overwrites TMEM that an earlier, still-running MMA reads.
//
// Rescaling is lazy: a row keeps its reference max until a tile raises the
// max by more than RESCALE_LOG2 (base-2 units); P and l always share the same
// reference, so O / l is unaffected and P stays below 2^RESCALE_LOG2.  Because
// the reference can sit below the row max, the dominant probability is not
// exactly 1 and its bf16 rounding would not cancel against an fp32 l; O is
// therefore divided by l~, the sum of the rounded probabilities (O is then an
// exact convex combination of the value rows), while the logsumexp uses l.
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
constexpr int NUM_THREADS = 192;
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr float RESCALE_LOG2 = 8.0f;

constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256, TM_P0 = 384, TM_P1 = 448;
constexpr uint32_t TM_COLS = 512;

// Device status word bits / wait codes.
constexpr uint32_t STATUS_TIMEOUT = 1u;

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
    static constexpr int DBLK = D / 64;                  // 64-element (128-byte) column blocks
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;     // one K or one V tile
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
    // barriers
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + STAGES;
    static constexpr int B_VFULL = B_KEMPTY + STAGES;
    static constexpr int B_VEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_VEMPTY + STAGES;  // 2
    static constexpr int B_PFULL = B_SFULL + 2;        // 2
    static constexpr int B_ODONE = B_PFULL + 2;        // 2
    static constexpr int B_DRAIN = B_ODONE + 2;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort
    static constexpr uint32_t USED = OFF_MISC + 16;
    static constexpr uint32_t SMEM_BYTES = USED + 1024;  // + slack to align the base to 1024
};

__device__ unsigned int g_status;      // STATUS_* bits, sticky until read by the host
__device__ unsigned int g_status_where;  // first wait code that gave up

// Wait codes: role * 256 + barrier index (+1 so that 0 means "none").
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
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(L::B_SFULL + b), 1);
            ptx::mbar_init(bar(L::B_PFULL + b), BM);
            ptx::mbar_init(bar(L::B_ODONE + b), 1);
        }
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
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
                ptx::tma_load_3d(sbase + L::OFF_Q + c * (BM * 128), &tm_q, bar(L::B_Q), c * 64, q0, bh);
            int nk = 0, nv = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % L::STAGES;
                const uint32_t ph = (uint32_t)(j / L::STAGES) & 1u;
                if (!wait_bar(bar(L::B_KEMPTY + s), ph ^ 1u, limit, abort_flag, 0x100 + L::B_KEMPTY + s)) break;
                ptx::mbar_arrive_expect_tx(bar(L::B_KFULL + s), L::KV_BYTES);
                for (int c = 0; c < L::DBLK; ++c)
                    ptx::tma_load_3d(sbase + L::OFF_K + s * L::KV_BYTES + c * (BN * 128), &tm_k,
                                     bar(L::B_KFULL + s), c * 64, j * BN, bh);
                ++nk;
                if (!wait_bar(bar(L::B_VEMPTY + s), ph ^ 1u, limit, abort_flag, 0x100 + L::B_VEMPTY + s)) break;
                ptx::mbar_arrive_expect_tx(bar(L::B_VFULL + s), L::KV_BYTES);
                for (int c = 0; c < L::DBLK; ++c)
                    ptx::tma_load_3d(sbase + L::OFF_V + s * L::KV_BYTES + c * (BN * 128), &tm_v,
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
            constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(BM, D, true);
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
                    const uint32_t koff = (uint32_t)(kk >> 2) * (BM * 128) + (uint32_t)(kk & 3) * 32;
                    const uint64_t a = ptx::sdesc_sw128(sbase + L::OFF_Q + koff, 16, 1024);
                    const uint64_t b = ptx::sdesc_sw128(
                        sbase + L::OFF_K + s * L::KV_BYTES + (uint32_t)(kk >> 2) * (BN * 128) +
                            (uint32_t)(kk & 3) * 32,
                        16, 1024);
                    ptx::mma_ss(d_tmem, a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(bar(L::B_KEMPTY + s));
                ptx::tc_commit(bar(L::B_SFULL + (j & 1)));
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n_kv > 1) ok = issue_s(1);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int b = j & 1;
                const int s = j % L::STAGES;
                if (!wait_bar(bar(L::B_PFULL + b), (uint32_t)(j >> 1) & 1u, limit, abort_flag,
                              0x200 + L::B_PFULL + b))
                    break;
                if (!wait_bar(bar(L::B_VFULL + s), (uint32_t)(j / L::STAGES) & 1u, limit, abort_flag,
                              0x200 + L::B_VFULL + s))
                    break;
                ptx::tc_fence_after_sync();
                // O (+)= P_j V_j: A = P from TMEM (2 bf16 per column, 8 columns per
                // 16 keys), B = V tile, MN-major (d contiguous): 64-wide d blocks
                // BN*128 bytes apart, 8-key groups 1024 bytes apart.
                const uint32_t p_tmem = tmem + (b ? TM_P1 : TM_P0);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bdesc = ptx::sdesc_sw128(
                        sbase + L::OFF_V + s * L::KV_BYTES + (uint32_t)kk * (16 * 128), BN * 128, 1024);
                    ptx::mma_ts(tmem + TM_O, p_tmem + (uint32_t)kk * 8, bdesc, IDESC_O,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::tc_commit(bar(L::B_VEMPTY + s));
                ptx::tc_commit(bar(L::B_ODONE + b));
                if (j + 2 < n_kv) ok = issue_s(j + 2);
            }
            // Drain: all MMAs issued by this thread complete before TMEM is freed.
            ptx::tc_commit(bar(L::B_DRAIN));
            drain_bar(bar(L::B_DRAIN), 0, limit, abort_flag, 0x280);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax warps
        const int row = threadIdx.x;  // 0..127 == TMEM lane
        const int q_idx = q0 + row;
        const int key_max = CAUSAL ? min(q_idx, N - 1) : N - 1;
        const int cta_key_max = CAUSAL ? min(q0, N - 1) : N - 1;  // smallest key_max of the CTA
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;
        float l = 0.f;   // sum of fp32 probabilities (logsumexp)
        float lr = 0.f;  // sum of the bf16-rounded probabilities (normalises O)
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            ok = warp_wait_bar(bar(L::B_SFULL + b), (uint32_t)(j >> 1) & 1u, limit, abort_flag,
                               0x300 + L::B_SFULL + b);
            if (!ok) break;
            ptx::tc_fence_after_sync();

            uint32_t r0[32], r1[32], r2[32], r3[32];
            const uint32_t s_tmem = tmem + lane_off + (b ? TM_S1 : TM_S0);
            ptx::tmem_ld32(s_tmem + 0, r0);
            ptx::tmem_ld32(s_tmem + 32, r1);
            ptx::tmem_ld32(s_tmem + 64, r2);
            ptx::tmem_ld32(s_tmem + 96, r3);
            ptx::tmem_wait_ld(r0);
            ptx::reg_fence(r1);
            ptx::reg_fence(r2);
            ptx::reg_fence(r3);
            float s[BN];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[c] = __uint_as_float(r0[c]);
                s[32 + c] = __uint_as_float(r1[c]);
                s[64 + c] = __uint_as_float(r2[c]);
                s[96 + c] = __uint_as_float(r3[c]);
            }
            // Causal diagonal tile / keys past N: -inf before the max.
            const int k0 = j * BN;
            if (k0 + BN - 1 > cta_key_max) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (k0 + c > key_max) s[c] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
            const float m_tile = mx * sl2;  // scale > 0, so max commutes with it

            if (j == 0) {
                m_ref = (m_tile == -INFINITY) ? 0.f : m_tile;
            } else {
                const float m_new = fmaxf(m_ref, m_tile);
                const bool need = m_new > m_ref + RESCALE_LOG2;
                if (__any_sync(0xffffffffu, need)) {
                    // O holds P_{j-1} V_{j-1} once that MMA is done; rescale it.
                    const int pb = (j - 1) & 1;
                    ok = warp_wait_bar(bar(L::B_ODONE + pb), (uint32_t)((j - 1) >> 1) & 1u, limit,
                                       abort_flag, 0x300 + L::B_ODONE + pb);
                    if (!ok) break;
                    ptx::tc_fence_after_sync();
                    const float corr = ptx::ex2(m_ref - m_new);
                    l *= corr;
                    lr *= corr;
                    m_ref = m_new;
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tmem + lane_off + TM_O + ch * 32, o);
                        ptx::tmem_wait_ld(o);
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
                        ptx::tmem_st32(tmem + lane_off + TM_O + ch * 32, o);
                    }
                    ptx::tmem_wait_st();
                }
            }

            // P = 2^(s*c - m_ref), rounded to bf16 for the P.V MMA.
            const float neg_m = -m_ref;
            uint32_t pk0[32], pk1[32];
            float rs0 = 0.f, rs1 = 0.f, rr0 = 0.f, rr1 = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float a0 = ptx::ex2(fmaf(s[2 * c], sl2, neg_m));
                const float a1 = ptx::ex2(fmaf(s[2 * c + 1], sl2, neg_m));
                const float b0 = ptx::ex2(fmaf(s[64 + 2 * c], sl2, neg_m));
                const float b1 = ptx::ex2(fmaf(s[64 + 2 * c + 1], sl2, neg_m));
                rs0 += a0 + a1;
                rs1 += b0 + b1;
                const uint32_t w0 = ptx::pack_bf16x2(a0, a1);
                const uint32_t w1 = ptx::pack_bf16x2(b0, b1);
                rr0 += __uint_as_float(w0 << 16) + __uint_as_float(w0 & 0xffff0000u);
                rr1 += __uint_as_float(w1 << 16) + __uint_as_float(w1 & 0xffff0000u);
                pk0[c] = w0;
                pk1[c] = w1;
            }
            l += rs0 + rs1;
            lr += rr0 + rr1;

            // P buffer b was last read by the MMA of tile j-2.
            if (j >= 2) {
                ok = warp_wait_bar(bar(L::B_ODONE + b), (uint32_t)((j - 2) >> 1) & 1u, limit, abort_flag,
                                   0x340 + L::B_ODONE + b);
                if (!ok) break;
                ptx::tc_fence_after_sync();
            }
            const uint32_t p_tmem = tmem + lane_off + (b ? TM_P1 : TM_P0);
            ptx::tmem_st32(p_tmem + 0, pk0);
            ptx::tmem_st32(p_tmem + 32, pk1);
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(L::B_PFULL + b));
        }

        // ------------------------------------------------------- epilogue
        if (ok) {
            const int lb = (n_kv - 1) & 1;
            ok = warp_wait_bar(bar(L::B_ODONE + lb), (uint32_t)((n_kv - 1) >> 1) & 1u, limit, abort_flag,
                               0x380 + L::B_ODONE + lb);
        }
        if (ok) {
            ptx::tc_fence_after_sync();
            const float inv_l = 1.0f / lr;
            // O row -> bf16 -> the Q tile's shared memory (Q is no longer read),
            // in the 128-byte-swizzled layout the O tensor map expects.
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                ptx::tmem_ld32(tmem + lane_off + TM_O + ch * 32, o);
                ptx::tmem_wait_ld(o);
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    w[c] = ptx::pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                            __uint_as_float(o[2 * c + 1]) * inv_l);
                const int col0 = ch * 32;
                const uint32_t blk = sbase + L::OFF_Q + (uint32_t)(col0 >> 6) * (BM * 128) + (uint32_t)row * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t chunk = (uint32_t)(((col0 & 63) >> 3) + u);
                    ptx::st_shared_v4(blk + ((chunk ^ (uint32_t)(row & 7)) << 4), w[4 * u], w[4 * u + 1],
                                      w[4 * u + 2], w[4 * u + 3]);
                }
            }
            if (q_idx < N)
                p.lse[(int64_t)bh * N + q_idx] = (m_ref + ptx::lg2(l)) * 0.69314718055994530942f;
        }
        ptx::fence_proxy_async_smem();
        ptx::named_barrier_sync(1, BM);
        if (threadIdx.x == 0 && *abort_flag == 0u) {
            for (int c = 0; c < L::DBLK; ++c)
                ptx::tma_store_3d(&tm_o, sbase + L::OFF_Q + c * (BM * 128), c * 64, q0, bh);
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
