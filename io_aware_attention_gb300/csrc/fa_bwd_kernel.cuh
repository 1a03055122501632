// Attention backward for sm_103a: tcgen05 tensor cores + TMEM + TMA.
//
// The gradients of O = softmax(scale * Q K^T (+ causal mask)) V for a given
// dO, with P recomputed tile by tile from the forward's logsumexp L instead of
// being stored ("Writing and Benchmarking Custom Kernels" §10.3.2):
//
//   D_i   = dO_i . O_i                                 (fa_bwd_prep_kernel)
//   P_ij  = 2^(S_ij * scale * log2 e - L_i * log2 e)   (S = Q K^T recomputed)
//   dV_j += sum_i P_ij dO_i
//   dP_ij = dO_i . V_j
//   dS_ij = P_ij (dP_ij - D_i)
//   dK_j += scale * sum_i dS_ij Q_i
//   dQ_i += scale * sum_j dS_ij K_j                    (fp32, added in L2)
//
// A work item is BKV = 128 keys of one (batch, head).  The item's K and V
// stay in shared memory while its query blocks of BQ = 64 rows stream
// through (under the causal mask only the blocks at or below the diagonal),
// and dK, dV accumulate in TMEM.  That is the loop order the page describes
// for the K/V gradient pass (query tiles inner), so dK and dV need no atomics;
// each step's dQ contribution is added into an fp32 accumulator in global
// memory with a TMA reduce-add (the add happens in L2), and fa_bwd_dq_kernel
// converts it at the end.
//
// Everything is computed transposed, keys on the TMEM lanes:
//   S^T  = K Q^T        (M = 128 keys, N = 64 queries, K = d)     smem x smem
//   dP^T = V dO^T       (same shape)                              smem x smem
//   dV  += P^T dO       (M = 128 keys, N = d, K = 64 queries)     TMEM x smem
//   dK  += dS^T Q       (same shape)                              smem x smem
//   dQ^T = K^T dS^T     (M = 128, N = 64 queries, K = 128 keys)   smem x smem
// so a thread of the P/dS warps owns one key row and P^T lands in TMEM in
// the layout the TS-form dV MMA reads as its A operand.  dS^T is written once
// to shared memory (128 rows of 128 bytes, 128-byte swizzle); the same bytes
// are the K-major A operand of the dK MMA and the MN-major B operand of the
// dQ MMA.  K is the MN-major A operand of the dQ MMA (K^T read in place).
// That MMA always has M = 128 (the TMEM lanes of a plain M = 128 product):
// for d = 64 its A operand is K's one 64-column block followed by a block of
// zeros kept in shared memory, so TMEM lanes 64-127 of dQ^T hold zeros and
// the dQ warps of those lanes skip the reduce.
//
// Warp roles (448 threads):
//   warps 0-7   P / dS.  Warp w serves keys 32*(w%4) .. +31 (its TMEM lane
//               quarter) and query columns 32*(w/4) .. +31 of every step.
//   warps 8-11  dQ: TMEM -> registers -> a shared-memory staging block ->
//               TMA reduce-add into the fp32 accumulator; at the end of an
//               item, the dK / dV epilogue.
//   warp 12     TMA producer: K, V once per item; Q and dO of each query
//               block into a ring of stages.
//   warp 13     MMA issuer (one elected lane); also allocates TMEM.
//
// TMEM columns (512): [0,64) S^T buffer 0, [64,128) S^T buffer 1 (P^T as bf16
// pairs is written over the first 16 columns of each 32-column half of its
// own buffer), [128,192) dP^T, [192,256) dQ^T, [256,256+d) dV, [384,384+d) dK.
//
// Shared memory is the tight resource.  An M = 128 MMA with both operands
// in shared memory reads them at the full 128 bytes per cycle of the SM (a
// 64-column MMA takes 48 cycles instead of 32), and while the tensor core
// does so every other shared-memory access queues behind it -- including
// mbarrier waits, which then take ~1000 cycles even on a completed phase.
// Hence:
//   - warps signal the MMA issuer through hardware named barriers (no shared
//     memory); mbarriers are left for what only they can carry: TMA byte
//     counts and MMA completion (tcgen05.commit);
//   - the issue order makes most completions implied: per step g
//         dV(g); [dP(g) read] S(g+1), dP(g+1); [dS(g) ready] dK(g); dQ(g)
//     The dP-read signal means dP(g) is complete, hence every MMA issued
//     before it, among them dV(g-1), the last reader of S(g+1)'s buffer;
//     dP(g+2) completing means dK(g) and dQ(g), the readers of dS buffer
//     g & 1, are complete;
//   - the P/dS warps take L*log2 e and D from global memory (L1/L2), loaded
//     at the top of a step, not from shared memory;
//   - the dQ contribution leaves through one bulk TMA reduce-add per warp and
//     step.  Per-element atomics from registers were tried: their thousands
//     of memory requests per step stall every warp's barrier operations
//     behind them (about 2000 cycles a step, against 150 for the staging
//     round trip);
//   - the Q/dO ring is three stages deep, released as soon as dK(g), its
//     last reader, is done.
//
// Named barriers are counted, not timed: every role executes each of its
// bar.arrive / bar.sync once per step (or item) whatever happened, so the
// counts always match.  mbarrier waits are bounded in time (see wait_bar);
// on expiry the CTA records the wait in the device status word and raises an
// abort flag, after which the roles keep walking their loops (skipping the
// work, still meeting the named barriers), drain in-flight copies / MMAs and
// reach the common exit, where TMEM is freed.  An aborted producer signals
// with bar.sync rather than bar.arrive (nb_signal), so it cannot run a
// generation ahead of the issuer; the issuer meets each producer group's
// barriers in the order that group signals them (P_READY, DP_READ, DS_READY
// per step; DQ_READ per step, then ACC_READ per item), so those syncs cannot
// wait on one another in a cycle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "fa_fwd_kernel.cuh"
#include "ptx.cuh"

namespace fa {
namespace bwd {

constexpr int BKV = 128;  // keys per work item (TMEM lanes)
constexpr int BQ = 64;    // query rows per step
constexpr int PDS_WARPS = 8;
constexpr int WARP_DQ0 = 8;  // warps 8..11
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA = 13;
constexpr int NUM_THREADS = 14 * 32;
constexpr int QSTAGES = 3;
constexpr uint32_t TM_S0 = 0, TM_S1 = 64, TM_DP = 128, TM_DQ = 192, TM_DV = 256, TM_DK = 384;
constexpr uint32_t TM_COLS = 512;

// Named barriers (0 is __syncthreads).  P/dS warps -> issuer: 256 + 32
// threads; dQ warps -> issuer: 128 + 32.  Each alternates between two ids by
// the parity of its step (or item): see nb_signal.
constexpr uint32_t NB_P_READY = 1;    // + (g & 1): P(g) in TMEM
constexpr uint32_t NB_DS_READY = 3;   // + (g & 1): dS(g) in shared memory
constexpr uint32_t NB_DP_READ = 5;    // + (g & 1): dP(g) read out of TMEM (so dP(g) is complete)
constexpr uint32_t NB_DQ_READ = 7;    // + (g & 1): dQ(g) read out of TMEM
constexpr uint32_t NB_ACC_READ = 9;   // + (k & 1): dK, dV of item k read out of TMEM
constexpr uint32_t NB_PDS_COUNT = 32 * PDS_WARPS + 32;
constexpr uint32_t NB_DQ_COUNT = 32 * 4 + 32;

// The producer warps signal with nb_signal (the forward kernel's header):
// bar.arrive while healthy, bar.sync after an abort.

struct Params {
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    const float* lse2;  // (B*H, Np): L * log2 e; +inf for rows >= N
    const float* dsum;  // (B*H, Np): D; 0 for rows >= N
    float* dq_acc;      // (B*H, Np, D): fp32 dQ / scale (D = the padded head size)
    int N;
    int d;         // the caller's head size (<= D, a multiple of 8): dK, dV row stride and stored columns
    int Np;        // query rows rounded up to a multiple of BQ
    int num_kb;    // key blocks per head
    int num_items; // B*H*num_kb
    float scale_log2;
    float scale;
    unsigned long long wait_limit_ns;
    int debug_skip_q;  // test hook: global step whose Q/dO tile the first CTA never loads (-1: none)
};

template <int D>
struct Layout {
    static_assert(D == 64 || D == 128, "head size");
    static constexpr uint32_t KV_BYTES = BKV * D * 2;   // K or V of an item (D / 64 64-column blocks)
    static constexpr uint32_t KBLK = BKV * 128;         // one 64-column block of K or V (16 KB)
    static constexpr uint32_t QT_BYTES = BQ * D * 2;    // a Q or dO tile
    static constexpr uint32_t QBLK = BQ * 128;          // one 64-column block of it (8 KB)
    static constexpr uint32_t DS_BYTES = BKV * BQ * 2;  // dS^T tile (128 rows x 128 B)
    static constexpr uint32_t STG_WARP = BQ * 32 * 4;   // one dQ warp's fp32 staging (64 x 32)
    static constexpr uint32_t OFF_K = 0;                // two blocks: K, or K and zeros when D = 64
    static constexpr uint32_t OFF_V = OFF_K + 2 * KBLK;
    static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;
    static constexpr uint32_t OFF_DO = OFF_Q + QSTAGES * QT_BYTES;
    static constexpr uint32_t OFF_DS = OFF_DO + QSTAGES * QT_BYTES;
    static constexpr uint32_t OFF_STG = OFF_DS + 2 * DS_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_STG + 4 * STG_WARP;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_KVEMPTY = 1;
    static constexpr int B_QFULL = 2;                   // QSTAGES
    static constexpr int B_QEMPTY = B_QFULL + QSTAGES;  // QSTAGES
    static constexpr int B_SFULL = B_QEMPTY + QSTAGES;  // 2 (per S buffer)
    static constexpr int B_DPFULL = B_SFULL + 2;
    static constexpr int B_DQFULL = B_DPFULL + 1;
    static constexpr int B_ACCFULL = B_DQFULL + 1;
    static constexpr int B_DRAIN = B_ACCFULL + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(OFF_Q % 1024 == 0 && OFF_DO % 1024 == 0 && OFF_DS % 1024 == 0, "swizzled tiles");
};

// Work item i -> (flattened head, key block).  Within a head the key blocks
// come light, heavy, light, heavy (kb = M-1, 0, M-2, 1, ...), and a CTA takes
// both items of a pair (2p, 2p+1): under the causal mask key block kb sees
// the query blocks from the diagonal on, so every pair costs about the same.
struct Item {
    int bh, key0, m0, nq;  // first key, first query block, query blocks
};

template <bool CAUSAL>
__device__ __forceinline__ Item item_of(int i, const Params& p)
{
    Item it;
    const int t = i % p.num_kb;
    const int kb = (t & 1) ? (t >> 1) : (p.num_kb - 1 - (t >> 1));
    it.bh = i / p.num_kb;
    it.key0 = kb * BKV;
    const int nqb = p.Np / BQ;
    it.m0 = CAUSAL ? it.key0 / BQ : 0;
    it.nq = nqb - it.m0;
    return it;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const Params p)
{
    using L = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t sbase = ptx::smem_addr(smem_raw);
    uint8_t* const sgen = smem_raw;
    if (sbase & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, STATUS_BAD_SMEM);
        return;
    }
    volatile uint32_t* const misc = reinterpret_cast<volatile uint32_t*>(sgen + L::OFF_MISC);
    volatile uint32_t* const abort_flag = misc + 1;
    auto bar = [&](int i) -> uint32_t { return sbase + L::OFF_BAR + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const int N = p.N;
    auto first_item = [&]() -> int { return 2 * (int)blockIdx.x; };
    auto next_item = [&](int i, int& step) -> int {
        ++step;
        return (step & 1) ? i + 1 : i - 1 + 2 * (int)gridDim.x;
    };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(L::B_KVFULL), 1);
        ptx::mbar_init(bar(L::B_KVEMPTY), 1);
        for (int s = 0; s < QSTAGES; ++s) {
            ptx::mbar_init(bar(L::B_QFULL + s), 1);
            ptx::mbar_init(bar(L::B_QEMPTY + s), 1);
        }
        ptx::mbar_init(bar(L::B_SFULL), 1);
        ptx::mbar_init(bar(L::B_SFULL + 1), 1);
        ptx::mbar_init(bar(L::B_DPFULL), 1);
        ptx::mbar_init(bar(L::B_DQFULL), 1);
        ptx::mbar_init(bar(L::B_ACCFULL), 1);
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == WARP_TMA && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_do);
        ptx::prefetch_tensormap(&tm_dq);
    }
    if (warp == WARP_MMA) {
        ptx::tmem_alloc(sbase + L::OFF_MISC, TM_COLS);
        ptx::tmem_relinquish();
    }
    if constexpr (D == 64) {
        // The zero block after K: head dims 64-127 of the dQ MMA's A operand.
        for (uint32_t i = threadIdx.x; i < L::KBLK / 16; i += NUM_THREADS)
            ptx::st_shared_v4(sbase + L::OFF_K + L::KBLK + 16u * i, 0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    if (warp == WARP_TMA) {
        // ---------------------------------------------------- TMA producer
        int g = 0, k = 0;
        bool ok = true;
        for (int i = first_item(), step = 0; ok && i < p.num_items; i = next_item(i, step), ++k) {
            const Item it = item_of<CAUSAL>(i, p);
            if (!(ok = warp_wait_bar(bar(L::B_KVEMPTY), (uint32_t)(k & 1) ^ 1u, limit, abort_flag,
                                     0x1100 + L::B_KVEMPTY)))
                break;
            if (ptx::elect_one()) {
                ptx::mbar_arrive_expect_tx(bar(L::B_KVFULL), 2 * L::KV_BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    ptx::tma_load_3d(sbase + L::OFF_K + c * L::KBLK, &tm_k, bar(L::B_KVFULL), c * 64, it.key0, it.bh);
                    ptx::tma_load_3d(sbase + L::OFF_V + c * L::KBLK, &tm_v, bar(L::B_KVFULL), c * 64, it.key0, it.bh);
                }
            }
            for (int t = 0; ok && t < it.nq; ++t, ++g) {
                const int s = g % QSTAGES;
                if (!(ok = warp_wait_bar(bar(L::B_QEMPTY + s), ((uint32_t)(g / QSTAGES) & 1u) ^ 1u, limit,
                                         abort_flag, 0x1100 + L::B_QEMPTY + s)))
                    break;
                // Test hook: the first CTA leaves one step's tile unloaded, so
                // the issuer's wait for it runs out (exercises the abort path).
                if (ptx::elect_one() && !(g == p.debug_skip_q && blockIdx.x == 0)) {
                    const int q0 = (it.m0 + t) * BQ;
                    const uint32_t fb = bar(L::B_QFULL + s);
                    ptx::mbar_arrive_expect_tx(fb, 2 * L::QT_BYTES);
                    for (int c = 0; c < D / 64; ++c) {
                        ptx::tma_load_3d(sbase + L::OFF_Q + s * L::QT_BYTES + c * L::QBLK, &tm_q, fb, c * 64, q0, it.bh);
                        ptx::tma_load_3d(sbase + L::OFF_DO + s * L::QT_BYTES + c * L::QBLK, &tm_do, fb, c * 64, q0,
                                         it.bh);
                    }
                }
            }
        }
        // Drain: every copy this warp issued lands before exit.
        if (k > 0) drain_bar(bar(L::B_KVFULL), (uint32_t)((k - 1) & 1), limit, abort_flag, 0x1180);
        for (int gg = max(0, g - QSTAGES); gg < g; ++gg)
            if (!(gg == p.debug_skip_q && blockIdx.x == 0))
                drain_bar(bar(L::B_QFULL + gg % QSTAGES), (uint32_t)(gg / QSTAGES) & 1u, limit, abort_flag, 0x1181);
    } else if (warp == WARP_MMA) {
        // ----------------------------------------------------- MMA issuer
        constexpr uint32_t ID_S = ptx::idesc_bf16_f32_ab(BKV, BQ, false, false);  // S^T, dP^T
        constexpr uint32_t ID_G = ptx::idesc_bf16_f32_ab(BKV, D, false, true);    // dV, dK
        constexpr uint32_t ID_Q = ptx::idesc_bf16_f32_ab(BKV, BQ, true, true);    // dQ^T (M = 128)
        // K-major descriptors (rows of 128 B, 8-row groups 1024 B apart).
        const uint64_t k_kmaj = ptx::sdesc_sw128(sbase + L::OFF_K, 16, 1024);
        const uint64_t v_kmaj = ptx::sdesc_sw128(sbase + L::OFF_V, 16, 1024);
        const uint64_t q_kmaj = ptx::sdesc_sw128(sbase + L::OFF_Q, 16, 1024);
        const uint64_t do_kmaj = ptx::sdesc_sw128(sbase + L::OFF_DO, 16, 1024);
        const uint64_t ds_kmaj = ptx::sdesc_sw128(sbase + L::OFF_DS, 16, 1024);
        // MN-major descriptors (64-element blocks LBO apart, 8-deep K groups 1024 B apart).
        const uint64_t k_mn = ptx::sdesc_sw128(sbase + L::OFF_K, L::KBLK, 1024);
        const uint64_t q_mn = ptx::sdesc_sw128(sbase + L::OFF_Q, L::QBLK, 1024);
        const uint64_t do_mn = ptx::sdesc_sw128(sbase + L::OFF_DO, L::QBLK, 1024);
        const uint64_t ds_mn = ptx::sdesc_sw128(sbase + L::OFF_DS, L::QBLK, 1024);
        auto off = [](uint32_t bytes) -> uint64_t { return (uint64_t)(bytes >> 4); };

        bool ok = true;
        // S^T(g) = K Q(g)^T into S buffer g & 1, then dP^T(g) = V dO(g)^T.
        // The caller has met the dP-read barrier of step g - 1, so every MMA
        // issued before dP(g-1) -- dV(g-2), the last reader of the S buffer --
        // is complete, and dP(g-1) has been read out.
        auto issue_s_dp = [&](int gg) {
            const int s = gg % QSTAGES, b = gg & 1;
            if (ok) ok = warp_wait_bar(bar(L::B_QFULL + s), (uint32_t)(gg / QSTAGES) & 1u, limit, abort_flag,
                                       0x1200 + L::B_QFULL + s);
            if (!ok) return;
            ptx::tc_fence_after_sync();
            const uint32_t d_tm = tmem + (b ? TM_S1 : TM_S0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (ptx::elect_one())
                    ptx::mma_ss(d_tm, k_kmaj + off((kk >> 2) * L::KBLK + (kk & 3) * 32),
                                q_kmaj + off(s * L::QT_BYTES + (kk >> 2) * L::QBLK + (kk & 3) * 32), ID_S,
                                kk > 0 ? 1u : 0u);
            }
            if (ptx::elect_one()) ptx::tc_commit(bar(L::B_SFULL + b));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (ptx::elect_one())
                    ptx::mma_ss(tmem + TM_DP, v_kmaj + off((kk >> 2) * L::KBLK + (kk & 3) * 32),
                                do_kmaj + off(s * L::QT_BYTES + (kk >> 2) * L::QBLK + (kk & 3) * 32), ID_S,
                                kk > 0 ? 1u : 0u);
            }
            if (ptx::elect_one()) ptx::tc_commit(bar(L::B_DPFULL));
        };

        int g = 0, k = 0;
        for (int i = first_item(), step = 0; i < p.num_items; i = next_item(i, step), ++k) {
            const Item it = item_of<CAUSAL>(i, p);
            if (ok) ok = warp_wait_bar(bar(L::B_KVFULL), (uint32_t)(k & 1), limit, abort_flag, 0x1200 + L::B_KVFULL);
            issue_s_dp(g);
            for (int t = 0; t < it.nq; ++t, ++g) {
                const int s = g % QSTAGES, b = g & 1;
                const bool more = t + 1 < it.nq;
                // dV += P^T dO: A = P^T from TMEM (bf16 pairs; queries 16kk.. at
                // column 32*(kk/2) + 8*(kk%2) of the S buffer), B = dO MN-major.
                // The first of an item overwrites dV: the epilogue has read it
                // (the dQ warps read the previous item's last dQ before that).
                if (t == 0 && k > 0) {
                    ptx::named_barrier_sync(NB_DQ_READ + (uint32_t)((g - 1) & 1), NB_DQ_COUNT);
                    ptx::named_barrier_sync(NB_ACC_READ + (uint32_t)((k - 1) & 1), NB_DQ_COUNT);
                }
                ptx::named_barrier_sync(NB_P_READY + (uint32_t)b, NB_PDS_COUNT);
                if (ok) {
                    ptx::tc_fence_after_sync();
                    const uint32_t p_tm = tmem + (b ? TM_S1 : TM_S0);
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk) {
                        if (ptx::elect_one())
                            ptx::mma_ts(tmem + TM_DV, p_tm + 32u * (kk >> 1) + 8u * (kk & 1),
                                        do_mn + off(s * L::QT_BYTES + kk * 2048), ID_G, (t > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                ptx::named_barrier_sync(NB_DP_READ + (uint32_t)b, NB_PDS_COUNT);  // dP(g) read
                if (more) issue_s_dp(g + 1);
                // dK += dS^T Q: A = dS^T K-major, B = Q MN-major.
                ptx::named_barrier_sync(NB_DS_READY + (uint32_t)b, NB_PDS_COUNT);
                if (ok) {
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk) {
                        if (ptx::elect_one())
                            ptx::mma_ss(tmem + TM_DK, ds_kmaj + off(b * L::DS_BYTES + kk * 32),
                                        q_mn + off(s * L::QT_BYTES + kk * 2048), ID_G, (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    // dK(g) is the stage's last reader (S, dP, dV came before it).
                    if (ptx::elect_one()) ptx::tc_commit(bar(L::B_QEMPTY + s));
                }
                // dQ^T = K^T dS^T: A = K MN-major, B = dS^T MN-major, once the
                // dQ warps have read dQ(g - 1) out of TMEM (at an item's first
                // step, met above).
                if (t > 0) ptx::named_barrier_sync(NB_DQ_READ + (uint32_t)((g - 1) & 1), NB_DQ_COUNT);
                if (ok) {
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < BKV / 16; ++kk) {
                        if (ptx::elect_one())
                            ptx::mma_ss(tmem + TM_DQ, k_mn + off(kk * 2048), ds_mn + off(b * L::DS_BYTES + kk * 2048),
                                        ID_Q, kk > 0 ? 1u : 0u);
                    }
                    if (ptx::elect_one()) {
                        ptx::tc_commit(bar(L::B_DQFULL));
                        if (!more) {
                            ptx::tc_commit(bar(L::B_ACCFULL));
                            ptx::tc_commit(bar(L::B_KVEMPTY));
                        }
                    }
                }
            }
        }
        // The last item's signals, so that every named barrier completes.
        if (k >= 1) {
            ptx::named_barrier_sync(NB_DQ_READ + (uint32_t)((g - 1) & 1), NB_DQ_COUNT);
            ptx::named_barrier_sync(NB_ACC_READ + (uint32_t)((k - 1) & 1), NB_DQ_COUNT);
        }
        if (ptx::elect_one()) ptx::tc_commit(bar(L::B_DRAIN));
        drain_bar(bar(L::B_DRAIN), 0, limit, abort_flag, 0x1280);
    } else if (warp >= WARP_DQ0) {
        // -------------------------------------------- dQ and the epilogue
        const int quarter = warp & 3;  // dQ^T lanes = head dims 32*quarter ..; dK/dV lanes = keys
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t stg = sbase + L::OFF_STG + quarter * L::STG_WARP;
        const bool has_dims = quarter * 32 < p.d;  // this lane quarter of dQ^T holds head dims
        int g = 0, k = 0;
        bool ok = true;
        for (int i = first_item(), step = 0; i < p.num_items; i = next_item(i, step), ++k) {
            const Item it = item_of<CAUSAL>(i, p);
            for (int t = 0; t < it.nq; ++t, ++g) {
                if (ok) ok = warp_wait_bar(bar(L::B_DQFULL), (uint32_t)g & 1u, limit, abort_flag, 0x1300 + L::B_DQFULL);
                // Every dQ warp waits for dQ(g) before it signals, so that no
                // warp runs a step ahead on the named barrier.
                if (ok && has_dims) {
                    uint32_t a[32], c[32];
                    ptx::tc_fence_after_sync();
                    ptx::tmem_ld32(tmem + lane_off + TM_DQ, a);
                    ptx::tmem_ld32(tmem + lane_off + TM_DQ + 32, c);
                    ptx::tmem_wait_ld(a);
                    ptx::reg_fence(c);
                    ptx::tc_fence_before_sync();
                    __syncwarp();
                    nb_signal(NB_DQ_READ + (uint32_t)(g & 1), NB_DQ_COUNT, ok);
                    // The staging block is free once this warp's previous reduce
                    // has read it.  Row q holds this warp's 32 head dims of query q.
                    if (lane == 0) ptx::tma_store_wait_read();
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(stg + q * 128 + lane * 4), "r"(a[q]) : "memory");
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(stg + (q + 32) * 128 + lane * 4), "r"(c[q])
                                     : "memory");
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_reduce_add_3d(&tm_dq, stg, quarter * 32, (it.m0 + t) * BQ, it.bh);
                        ptx::tma_store_commit();
                    }
                } else {
                    __syncwarp();
                    nb_signal(NB_DQ_READ + (uint32_t)(g & 1), NB_DQ_COUNT, ok);
                }
            }
            // Epilogue: dV and scale * dK of this warp's 32 keys, bf16.
            if (ok) ok = warp_wait_bar(bar(L::B_ACCFULL), (uint32_t)k & 1u, limit, abort_flag, 0x1300 + L::B_ACCFULL);
            if (ok) {
                ptx::tc_fence_after_sync();
                const int key = it.key0 + quarter * 32 + lane;
                const bool key_ok = key < N;
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    __nv_bfloat16* const dst = (which ? p.dk : p.dv) + ((int64_t)it.bh * N + key) * p.d;
                    const float mul = which ? p.scale : 1.0f;
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tmem + lane_off + (which ? TM_DK : TM_DV) + ch * 32, o);
                        ptx::tmem_wait_ld(o);
                        uint32_t w[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            w[c] = ptx::pack_bf16x2(__uint_as_float(o[2 * c]) * mul, __uint_as_float(o[2 * c + 1]) * mul);
                        if (key_ok) {
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                if (ch * 32 + u * 8 < p.d)
                                    ptx::st_global_v4(dst + ch * 32 + u * 8, w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                      w[4 * u + 3]);
                        }
                    }
                }
                ptx::tc_fence_before_sync();
            }
            __syncwarp();
            nb_signal(NB_ACC_READ + (uint32_t)(k & 1), NB_DQ_COUNT, ok);
        }
        // Every reduce this warp issued completes before exit.
        if (lane == 0) ptx::bulk_wait_all();
        __syncwarp();
    } else {
        // ------------------------------------------------------ P / dS warps
        const int quarter = warp & 3;
        const int half = warp >> 2;          // query columns 32*half .. +31 of a step
        const int r = quarter * 32 + lane;   // key row in the item == TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        int g = 0;
        bool ok = true;
        for (int i = first_item(), step = 0; i < p.num_items; i = next_item(i, step)) {
            const Item it = item_of<CAUSAL>(i, p);
            const int key = it.key0 + r;
            const bool key_ok = key < N;
            for (int t = 0; t < it.nq; ++t, ++g) {
                const int b = g & 1;
                const int q0 = (it.m0 + t) * BQ + half * 32;  // first query of this thread's columns
                // L*log2 e and D of this thread's 32 queries, loaded before the waits.
                const float4* const lrow = reinterpret_cast<const float4*>(p.lse2 + (int64_t)it.bh * p.Np + q0);
                const float4* const drow = reinterpret_cast<const float4*>(p.dsum + (int64_t)it.bh * p.Np + q0);
                float4 l4[8], d4[8];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) l4[c4] = __ldg(lrow + c4);

                if (ok) ok = warp_wait_bar(bar(L::B_SFULL + b), (uint32_t)(g >> 1) & 1u, limit, abort_flag,
                                           0x1400 + L::B_SFULL + b);
                const uint32_t s_tm = tmem + lane_off + (b ? TM_S1 : TM_S0) + 32u * half;
                // The scores, then (in place) P as fp32 bit patterns.
                uint32_t pv[32];
                if (!ok) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) pv[c] = 0u;
                } else {
                    ptx::tc_fence_after_sync();
                    ptx::tmem_ld32(s_tm, pv);
                    ptx::tmem_wait_ld(pv);
                    // P = 2^(s * scale * log2 e - L * log2 e); masked entries 0.
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        pv[4 * c4 + 0] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pv[4 * c4 + 0]), sl2, -l4[c4].x)));
                        pv[4 * c4 + 1] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pv[4 * c4 + 1]), sl2, -l4[c4].y)));
                        pv[4 * c4 + 2] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pv[4 * c4 + 2]), sl2, -l4[c4].z)));
                        pv[4 * c4 + 3] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pv[4 * c4 + 3]), sl2, -l4[c4].w)));
                    }
                    if (!key_ok) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) pv[c] = 0u;
                    } else if (CAUSAL && q0 < it.key0 + BKV - 1) {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (q0 + c < key) pv[c] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[c] = ptx::pack_bf16x2(__uint_as_float(pv[2 * c]), __uint_as_float(pv[2 * c + 1]));
                    ptx::tmem_st16(s_tm, pk);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before_sync();
                }
                __syncwarp();
                nb_signal(NB_P_READY + (uint32_t)b, NB_PDS_COUNT, ok);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) d4[c4] = __ldg(drow + c4);

                // dP(g).  Its completion also means dK(g-2) and dQ(g-2), the
                // readers of dS buffer b, are done (they were issued before it).
                if (ok) ok = warp_wait_bar(bar(L::B_DPFULL), (uint32_t)g & 1u, limit, abort_flag, 0x1400 + L::B_DPFULL);
                uint32_t dp[32];
                if (!ok) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) dp[c] = 0u;
                } else {
                    ptx::tc_fence_after_sync();
                    ptx::tmem_ld32(tmem + lane_off + TM_DP + 32u * half, dp);
                    ptx::tmem_wait_ld(dp);
                    ptx::tc_fence_before_sync();
                }
                __syncwarp();
                nb_signal(NB_DP_READ + (uint32_t)b, NB_PDS_COUNT, ok);
                if (ok) {
                    // dS = P (dP - D), bf16 pairs, into dS^T buffer b (row r,
                    // bytes 64*half .. +63, 128-byte swizzle: 16-byte chunk c of
                    // row r sits at chunk c ^ (r & 7)).
                    uint32_t dk2[16];
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float e0 = __uint_as_float(pv[4 * c4 + 0]) * (__uint_as_float(dp[4 * c4 + 0]) - d4[c4].x);
                        const float e1 = __uint_as_float(pv[4 * c4 + 1]) * (__uint_as_float(dp[4 * c4 + 1]) - d4[c4].y);
                        const float e2 = __uint_as_float(pv[4 * c4 + 2]) * (__uint_as_float(dp[4 * c4 + 2]) - d4[c4].z);
                        const float e3 = __uint_as_float(pv[4 * c4 + 3]) * (__uint_as_float(dp[4 * c4 + 3]) - d4[c4].w);
                        dk2[2 * c4] = ptx::pack_bf16x2(e0, e1);
                        dk2[2 * c4 + 1] = ptx::pack_bf16x2(e2, e3);
                    }
                    const uint32_t row_addr = sbase + L::OFF_DS + b * L::DS_BYTES + (uint32_t)r * 128u;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t chunk = (uint32_t)(half * 4 + u) ^ (uint32_t)(r & 7);
                        ptx::st_shared_v4(row_addr + chunk * 16u, dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2],
                                          dk2[4 * u + 3]);
                    }
                    ptx::fence_proxy_async_smem();
                }
                __syncwarp();
                nb_signal(NB_DS_READY + (uint32_t)b, NB_PDS_COUNT, ok);
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

// D_i = dO_i . O_i and L_i * log2 e for every row i < Np of every head (rows
// >= N: D = 0, L * log2 e = +inf, so their recomputed P is 0), and the fp32
// dQ accumulator (Dp floats a row) zeroed.  A warp takes PREP_ROWS
// consecutive rows (one head's: Np is a multiple of 64) and issues all their
// loads before it reduces any, so that enough bytes are in flight; lane l
// takes elements 8l .. 8l + 7 of a row (d <= 128).
constexpr int PREP_ROWS = 4;

__global__ void __launch_bounds__(256, 4)
    fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                       const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ dsum,
                       float* __restrict__ dq_acc, int N, int Np, int d, int Dp, int64_t rows)
{
    const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * PREP_ROWS;
    const int lane = threadIdx.x & 31;
    if (row0 >= rows) return;
    const int64_t bh = row0 / Np;
    const int i0 = (int)(row0 - bh * Np);
    const int c = lane * 8;
    const __nv_bfloat16* const po = o + (bh * N + i0) * d + c;
    const __nv_bfloat16* const pd = dout + (bh * N + i0) * d + c;
    uint4 a[PREP_ROWS], b[PREP_ROWS];
#pragma unroll
    for (int r = 0; r < PREP_ROWS; ++r) {
        a[r] = b[r] = make_uint4(0u, 0u, 0u, 0u);
        if (i0 + r < N && c < d) {
            a[r] = *reinterpret_cast<const uint4*>(po + r * d);
            b[r] = *reinterpret_cast<const uint4*>(pd + r * d);
        }
    }
    float acc[PREP_ROWS];
#pragma unroll
    for (int r = 0; r < PREP_ROWS; ++r) {
        const uint32_t aw[4] = {a[r].x, a[r].y, a[r].z, a[r].w}, bw[4] = {b[r].x, b[r].y, b[r].z, b[r].w};
        acc[r] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[j]));
            const float2 bf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[j]));
            acc[r] = fmaf(af.x, bf.x, acc[r]);
            acc[r] = fmaf(af.y, bf.y, acc[r]);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], m);
    }
    if (lane < PREP_ROWS) {
        float v = acc[0];
#pragma unroll
        for (int r = 1; r < PREP_ROWS; ++r)
            if (lane == r) v = acc[r];
        const int i = i0 + lane;
        dsum[row0 + lane] = i < N ? v : 0.f;
        lse2[row0 + lane] = i < N ? lse[bh * N + i] * 1.4426950408889634074f : __int_as_float(0x7f800000);
    }
    // The warp's rows are consecutive: one block of PREP_ROWS * Dp floats.
    float4* const z = reinterpret_cast<float4*>(dq_acc + row0 * Dp);
    for (int k = lane; k < PREP_ROWS * Dp / 4; k += 32) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator) for rows < N; the accumulator is
// (B*H, Np, Dp), dQ (B*H, N, d).  Each thread converts 8 consecutive elements.
__global__ void __launch_bounds__(256)
    fa_bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, int N, int Np, int d,
                     int Dp, int64_t n8, float scale)
{
    const int64_t e8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e8 >= n8) return;
    const int64_t e = e8 * 8;
    const int64_t row = e / d;  // bh * N + i
    const int col = (int)(e - row * d);
    const int64_t bh = row / N;
    const int64_t i = row - bh * N;
    const float4* const src = reinterpret_cast<const float4*>(dq_acc + (bh * Np + i) * Dp + col);
    const float4 a = src[0], b = src[1];
    uint4 w;
    w.x = ptx::pack_bf16x2(a.x * scale, a.y * scale);
    w.y = ptx::pack_bf16x2(a.z * scale, a.w * scale);
    w.z = ptx::pack_bf16x2(b.x * scale, b.y * scale);
    w.w = ptx::pack_bf16x2(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(dq + e) = w;
}

}  // namespace bwd
}  // namespace fa
