// Attention forward for sm_103a: tcgen05 tensor cores + TMEM + TMA.
//
// A work item is BM = 128 query rows of one (batch, head).  Its key / value
// rows stream through shared memory in tiles of BN = 128 while an
// online-softmax state is carried per row ("Kernels — fusion and
// FlashAttention" §3–§4; "Fusion and IO-aware kernels" § FlashAttention,
// steps 1–4):
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
// The kernel is persistent: one CTA per SM takes work items i = blockIdx.x,
// blockIdx.x + gridDim.x, ... (query blocks of a head next to each other, so a
// head's K/V stay in L2 while its blocks run).  The pipelines run on across
// items: the next item's Q load and first score MMAs overlap the current
// item's last tiles and epilogue.
//
// Warp roles (512 threads):
//   warps 0-7  softmax.  Warp w serves query rows 32*(w%4) .. +31 (its TMEM
//              lane quarter) and score columns 64*(w/4) .. +63, so every SM
//              sub-partition runs two softmax warps (w and w+4, the two halves
//              of the same rows).  Each thread owns half a row: masking,
//              partial row max (returned with the scores by the TMEM load
//              itself, tcgen05.ld.red, and exchanged with the partner warp
//              through TMEM and a 64-thread named barrier), exponentials, its half of
//              P and its half of the O columns for rescaling.  At the end of
//              an item it leaves its reference max and row sum in TMEM for
//              the epilogue warps and goes straight on to the next item.
//   warps 8-11 epilogue, warp 8 + q for TMEM lane quarter q: once an item's
//              last P.V is complete, O / l~ and the logsumexp of its rows,
//              from TMEM to global memory.  The softmax warps issue no global
//              stores at all: their barriers (bar.sync, mbarrier arrive with
//              release semantics) would otherwise wait for those stores to
//              complete, a long stall at every item boundary.
//   warp 12    TMA producer of Q (once per item) and K_j (a ring of stages).
//   warp 13    score MMA issuer (S_j = Q K_j^T); also allocates TMEM.
//   warp 14    P.V MMA issuer.
//   warp 15    TMA producer of V_j (a ring of stages).
//   The issuers are converged warps; one elected lane issues each copy, MMA
//   and commit.  Two MMA issuers on two sub-partitions halve the instruction
//   stream each must get through per tile while the softmax warps' exponent
//   loops take most of the issue slots.  Registers: the CTA is launched with
//   128 a thread; the two softmax warpgroups raise theirs to 168 (D = 128;
//   152 at D = 64) and the other two lower theirs to 88 (104) (setmaxnreg),
//   which adds up to the register file.
//
// TMEM columns (512 allocated, lanes = query rows):
//   [  0,128) S buffer 0     [128,256) S buffer 1   (fp32 scores, double-buffered)
//   [256,256+d) O (fp32)     [256+d, 256+d+16) l~ (16 equal copies)
//   [400,464) P (bf16 pairs, one tile)
//   [468,472) the two halves' row maxima of a tile, per S buffer
//   [472,480) two statistics slots (item parity), each m_0, m_1, l_0, l_1: the
//             halves' reference maxima and fp32 row sums for the epilogue
// S_{j+2} goes into S_j's buffer as soon as every softmax warp has read S_j
// into registers (S_READ); P_j goes into the P buffer once P_{j-1} V_{j-1} is
// complete (O_DONE).  So the score stream runs ahead of the P.V stream and
// neither issuer waits for the other.  The score issuer hands "S_j written"
// to the softmax warps through a named barrier (see its loop).
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
// D = 64 runs a split design (Layout<64>::SPLIT).  Each row is carried as two
// independent halves h = 0, 1 (keys 64h .. 64h+63 of every tile, the warps w
// and w+4 of a lane quarter), each with its own reference max m_h, row sum
// l_h, P written over its half of the S buffer, and accumulator
// [O_h | l~_h] = sum over tiles of P_h [V_h | 1] (TMEM: S 2 x 128 columns,
// [O_h | l~_h] 2 x 80).  The halves merge once per item in the epilogue by
// their maxima, as split-key partial results do: with w_h = 2^(m_h - M),
// M = max(m_0, m_1), out = (w_0 O_0 + w_1 O_1) / (w_0 l~_0 + w_1 l~_1) and
// lse = (M + log2(w_0 l_0 + w_1 l_1)) ln 2.  The two warps of a row then never
// wait for each other inside the tile loop, which pays where the softmax
// bounds the kernel (d = 64: half the tensor work per tile).  At D = 128 the
// two [O_h | l~_h] accumulators do not fit next to the S buffers.
//
// Head sizes d < D (multiples of 8) run in the D = 64 or 128 instance: the
// TMA boxes are 64 columns wide and fill columns past d with zeros, which add
// nothing to any dot product; the epilogue stores d columns with row stride d.
//
// Every mbarrier wait is bounded in time; on expiry the thread records the
// wait in the device status word, raises a CTA-wide abort flag, and all roles
// drain their in-flight copies / MMAs and reach the common exit, where TMEM is
// freed.  Named barriers are counted, not timed: the roles that meet them
// (score issuer, softmax warps) walk every item and tile also after an abort,
// skipping the work, so every generation completes.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fa {

constexpr int BM = 128;  // query rows per work item
constexpr int BN = 128;  // keys per K/V tile
constexpr int SOFTMAX_THREADS = 256;
constexpr int SOFTMAX_WARPS = SOFTMAX_THREADS / 32;
constexpr int WARP_EPI0 = 8;  // warps 8-11: the epilogue, one per TMEM lane quarter
constexpr int EPI_WARPS = 4;
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA_S = 13;
constexpr int WARP_MMA_O = 14;
constexpr int WARP_TMA_V = 15;
constexpr int NUM_THREADS = 16 * 32;
// Registers a thread after the split (launched with 65536 / 512 = 128): the
// softmax warpgroups take REGS_SOFTMAX, the other two REGS_OTHER (per head
// size, in Layout): 168 / 88 at D = 128, 152 / 104 at D = 64, where the
// epilogue warps hold a whole row of the split design and the softmax needs
// fewer; 256 * (168 + 88) = 256 * (152 + 104) = 65536.
constexpr float RESCALE_LOG2 = 8.0f;
constexpr uint32_t WAIT_SLEEP_NS = 20000;  // suspend-time hint of one poll
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256, TM_P = 400, TM_MX = 468, TM_ST = 472;
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t BLK_BYTES = BN * 128;  // one 64-column, 128-row swizzled block (16 KB)

constexpr uint32_t STATUS_TIMEOUT = 1u;
constexpr uint32_t STATUS_BAD_SMEM = 2u;

// Named barriers (0 is __syncthreads): 1..4 pair the two softmax warps of a
// lane quarter; 5..7 carry "S of tile g is in TMEM" from the score MMA issuer
// to the softmax warps, id 5 + g % 3 (see nb_signal: the score stream runs
// two tiles ahead, so a generation's id may come round again only after two
// others).
constexpr uint32_t NB_PAIR0 = 1;
constexpr uint32_t NB_SREADY0 = 5;  // + (g % 3)
constexpr uint32_t NB_SREADY_COUNT = SOFTMAX_THREADS + 32;
// The split design (D = 64): one S-ready signal per half-row group, id
// 5 + 3h + g % 3, met by that group's four warps and the score issuer.
constexpr uint32_t NB_SREADY_SPLIT0 = 5;
constexpr uint32_t NB_SREADY_SPLIT_COUNT = SOFTMAX_THREADS / 2 + 32;

// Producer side of a producer -> consumers named barrier; the consumers meet
// every generation with bar.sync, in order.  While the pipeline runs, the
// producer only arrives (bar.arrive does not wait), and the mbarrier it
// waited on before signalling generation n guarantees that generation n - P
// has completed (P, the pacing depth, is 1 for the backward's signals and 2
// for the forward's S-ready signal).  After an abort those waits are
// skipped, so the producer joins with bar.sync instead.  Generation n uses id
// base + n % (P + 1): then, when the producer arrives for generation n, the
// generation that last used the id, n - P - 1, has completed -- through the
// mbarrier wait of the arrival before, or through the bar.sync it went
// through -- even when it switched from arriving to syncing in between.
// (With fewer ids, an aborted producer's sync could land on a generation
// that its own earlier arrival has not seen complete yet.)
__device__ __forceinline__ void nb_signal(uint32_t id, uint32_t count, bool ok)
{
    if (ok)
        ptx::named_barrier_arrive(id, count);
    else
        ptx::named_barrier_sync(id, count);
}

struct Params {
    __nv_bfloat16* o;
    float* lse;
    int N;
    int d;  // the caller's head size (<= D, a multiple of 8): O's row stride and stored columns
    int num_m_blocks;
    int num_bh;        // B * H
    int num_items;
    float scale_log2;  // scale * log2(e)
    unsigned long long wait_limit_ns;
    int debug_skip_k;  // test hook: global K tile the producer never loads (-1: none)
};

template <int D>
struct Layout {
    static_assert(D == 64 || D == 128, "head size");
    // D = 64 runs the split design: the two half-row warps of a row keep
    // separate softmax states and accumulators [O_h | l~_h] (TMEM has room
    // for both at D = 64) and merge them in the epilogue.
    static constexpr bool SPLIT = D == 64;
    static constexpr uint32_t REGS_SOFTMAX = (D == 64) ? 152 : 168;
    static constexpr uint32_t REGS_OTHER = (D == 64) ? 104 : 88;
    static_assert(SOFTMAX_THREADS * REGS_SOFTMAX + (NUM_THREADS - SOFTMAX_THREADS) * REGS_OTHER <= 65536,
                  "register split");
    static constexpr uint32_t O_STRIDE = D + 16;  // split design: O_1 follows [O_0 | l~_0]
    static constexpr int KSTAGES = (D == 128) ? 3 : 4;  // K runs two tiles ahead of V
    static constexpr int VSTAGES = (D == 128) ? 2 : 4;
    static constexpr int DBLK = D / 64;                   // 64-column blocks of a row
    static constexpr uint32_t TM_L = TM_O + D;            // l~ columns
    static_assert(TM_L + 16 <= TM_P && TM_P + 64 <= TM_MX && TM_MX + 4 <= TM_ST && TM_ST + 8 <= TM_COLS,
                  "TMEM budget");
    static_assert(!SPLIT || TM_O + 2 * O_STRIDE <= TM_ST, "TMEM budget (split)");
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;      // bytes of one K or V tile
    static constexpr uint32_t VSTAGE = (DBLK + 1) * BLK_BYTES;  // V blocks + the ones block
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KSTAGES * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + VSTAGES * VSTAGE;
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = 1;
    static constexpr int B_KFULL = 2;
    static constexpr int B_KEMPTY = B_KFULL + KSTAGES;
    static constexpr int B_VFULL = B_KEMPTY + KSTAGES;
    static constexpr int B_VEMPTY = B_VFULL + VSTAGES;
    static constexpr int B_SFULL = B_VEMPTY + VSTAGES;  // 2 (per S buffer): S written
    static constexpr int B_SREAD = B_SFULL + 2;         // 2 (per S buffer): S read out (one-state design)
    static constexpr int B_PFULL = B_SREAD + 2;         // P written; split: 4 (2 * half + S buffer)
    static constexpr int B_ODONE = B_PFULL + 4;  // every P.V; split: 2 (per S buffer, both halves)
    static constexpr int B_OFINAL = B_ODONE + 2; // the last P.V of an item
    static constexpr int B_OFREE = B_OFINAL + 1;
    static constexpr int B_DRAIN = B_OFREE + 1;  // 2 (one per MMA issuer)
    static constexpr int B_STFULL = B_DRAIN + 2;  // 2 (per stats slot): the softmax warps wrote it
    static constexpr int B_STFREE = B_STFULL + 2; // 2 (per stats slot): the epilogue warps read it (split design)
    static constexpr int NUM_BARS = B_STFREE + 2;
    static constexpr uint32_t OFF_MISC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;  // [0] TMEM base, [1] abort
    // The dynamic shared memory base is 1024-byte aligned (no static shared
    // memory); the kernel checks it and refuses to run otherwise.
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ unsigned int g_status;        // STATUS_* bits, sticky until read by the host
__device__ unsigned int g_status_where;  // first wait code that gave up (+1)

// Optional event trace for pipeline studies (compiled only with FA_TRACE):
// clock64() stamps of selected events of the first TRACE_CTAS CTAs, written to
// g_trace[cta][role][tile * 8 + event] for tiles < TRACE_TILES; role = warp
// index (softmax warps 0-7, epilogue 8-11, producer 12, MMA issuers 13 and 14); tile counts all tiles
// the CTA processed so far.
#ifdef FA_TRACE
constexpr int TRACE_CTAS = 8, TRACE_ROLES = 16, TRACE_TILES = 64;
__device__ unsigned long long* g_trace;
#define FA_TRACE_EV(role, tile, ev)                                                                  \
    do {                                                                                             \
        if (trace_buf && (tile) >= 0 && (tile) < TRACE_TILES)                                        \
            trace_buf[((size_t)blockIdx.x * TRACE_ROLES + (role)) * (TRACE_TILES * 8) + (tile) * 8 + (ev)] = \
                clock64();                                                                           \
    } while (0)
#else
#define FA_TRACE_EV(role, tile, ev) \
    do {                            \
    } while (0)
#endif

__device__ __forceinline__ void record_timeout(uint32_t code, volatile uint32_t* abort_flag)
{
    *abort_flag = 1u;
    atomicCAS(&g_status_where, 0u, code + 1u);
    atomicOr(&g_status, STATUS_TIMEOUT);
}

// Bounded wait on an mbarrier phase.  Gives up (returns false) when the CTA
// has aborted or after `limit_ns`, in which case it raises the abort.  The
// abort flag and the clock are looked at only every 256 polls.  A waiting
// thread sleeps in try_wait (woken when the phase completes) rather than
// spinning: a spinning warp takes issue slots from the warps on its SM
// sub-partition, among them the MMA issuers.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                         volatile uint32_t* abort_flag, uint32_t code)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = 0;
    for (uint32_t polls = 1;; ++polls) {
        if (ptx::mbar_try_wait_sleep(bar, parity, WAIT_SLEEP_NS)) return true;
        if ((polls & 255u) == 0u) {
            if (*abort_flag) return false;
            const uint64_t t = ptx::globaltimer_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > limit_ns) {
                record_timeout(code, abort_flag);
                return false;
            }
        }
    }
}

// Bounded wait used while draining: ignores the abort flag (in-flight copies
// must land before the CTA exits) but still gives up after `limit_ns`.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile uint32_t* abort_flag, uint32_t code)
{
    uint64_t t0 = 0;
    for (uint32_t polls = 0; !ptx::mbar_try_wait(bar, parity); ++polls) {
        if ((polls & 255u) == 255u) {
            const uint64_t t = ptx::globaltimer_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > limit_ns) {
                record_timeout(code, abort_flag);
                return;
            }
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

// Max of 64 values (fp32 bit patterns) with 3-input max instructions (depth 4).
__device__ __forceinline__ float max64(const uint32_t (&s)[64])
{
    float t[22];
#pragma unroll
    for (int i = 0; i < 21; ++i)
        t[i] = ptx::fmax3(__uint_as_float(s[3 * i]), __uint_as_float(s[3 * i + 1]), __uint_as_float(s[3 * i + 2]));
    t[21] = __uint_as_float(s[63]);
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
#pragma unroll
    for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t o[32];
        ptx::tmem_ld32(taddr + ch * 32, o);
        ptx::tmem_wait_ld(o);
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
        ptx::tmem_st32(taddr + ch * 32, o);
    }
}

// Multiplies this thread's D columns of an O accumulator (TMEM, from `taddr`)
// by `corr` (the split design).
template <int D>
__device__ __forceinline__ void scale_row(uint32_t taddr, float corr)
{
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        ptx::tmem_ld32(taddr + ch * 32, o);
        ptx::tmem_wait_ld(o);
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
        ptx::tmem_st32(taddr + ch * 32, o);
    }
}

// Stores the 32 words (eight 16-byte chunks, 128 bytes) of one row that each
// lane of a warp holds -- lane l holds row l; rows are `stride` elements apart
// from `base` -- so that every store instruction writes whole 128-byte lines:
// within each group of 8 lanes, the 8 x 8 matrix of chunks (lane = row, chunk
// = column) is transposed by three butterfly stages of shuffles, after which
// lane j of group g holds chunk j of rows 8g .. 8g+7.  A warp then stores 4
// lines per instruction, where the rows straight from registers would touch
// 32 lines per instruction and hold up the SM's memory pipeline.  Rows >=
// rows_left are not stored.
__device__ __forceinline__ void store_rows_coalesced(uint32_t (&w)[32], __nv_bfloat16* base, int lane, int rows_left,
                                                     int stride)
{
    const int j = lane & 7;
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) {
        const bool up = (j & s) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i & s) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t send = up ? w[4 * i + c] : w[4 * (i | s) + c];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, s);
                if (up)
                    w[4 * i + c] = recv;
                else
                    w[4 * (i | s) + c] = recv;
            }
        }
    }
    const int g = lane >> 3;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * g + i;
        if (r < rows_left)
            ptx::st_global_v4(base + (int64_t)r * stride + j * 8, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// Work item i: (flattened head, query block).  Two static orders:
//  - pairs (SNAKE == false): within a head the blocks come heavy, light, heavy,
//    light (m = M-1, 0, M-2, 1, ...), and a CTA always takes the two items of
//    a pair (2p, 2p+1): under the causal mask every pair then costs the same
//    M + 1 key tiles, and a head's blocks run at the same time on
//    neighbouring SMs, so its K/V are read from L2;
//  - by cost (SNAKE, causal problems whose K and V fit in L2): item
//    rank r is query block M - 1 - r / BH of head r % BH (heaviest first), and
//    CTA c takes ranks c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... (G CTAs): with
//    fewer pairs than a few per CTA, this balances far better.  A rank is
//    turned into the item's index in the pair order (item_of_rank), so that
//    item_of serves both.
struct Item {
    int bh, q0, n_kv;
};

// Index (in the pair order) of the item of cost rank r; num_items once the
// ranks are exhausted.
__device__ __forceinline__ int item_of_rank(int r, const Params& p)
{
    if (r >= p.num_items) return p.num_items;
    const int M = p.num_m_blocks;
    const int level = r / p.num_bh;
    const int bh = r - level * p.num_bh;
    const int m = M - 1 - level;
    const int t = (2 * (M - 1 - m) < M) ? 2 * (M - 1 - m) : 2 * m + 1;
    return bh * M + t;
}

template <bool CAUSAL>
__device__ __forceinline__ Item item_of(int i, const Params& p)
{
    Item it;
    const int t = i % p.num_m_blocks;
    const int m_block = (t & 1) ? (t >> 1) : (p.num_m_blocks - 1 - (t >> 1));
    it.bh = i / p.num_m_blocks;
    it.q0 = m_block * BM;
    const int n_kv_all = (p.N + BN - 1) / BN;
    it.n_kv = CAUSAL ? min(n_kv_all, (it.q0 + BM - 1) / BN + 1) : n_kv_all;
    return it;
}

// PAD: the caller's head size p.d is below D (stores are guarded and strided
// by p.d); the instances for d = D compile without the guard.  SNAKE: the
// items run in cost order (see item_of).
template <int D, bool CAUSAL, bool PAD, bool SNAKE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    using L = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t sbase = ptx::smem_addr(smem_raw);
    uint8_t* const sgen = smem_raw;
    if (sbase & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
        if (threadIdx.x == 0) atomicOr(&g_status, STATUS_BAD_SMEM);
        return;  // uniform: every thread leaves before any barrier or TMEM use
    }
    volatile uint32_t* const misc = reinterpret_cast<volatile uint32_t*>(sgen + L::OFF_MISC);
    volatile uint32_t* const abort_flag = misc + 1;
    auto bar = [&](int i) -> uint32_t { return sbase + L::OFF_BAR + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const int N = p.N;
    // This CTA's items (see item_of): pairs p = blockIdx.x, blockIdx.x +
    // gridDim.x, ..., both items 2p and 2p + 1 of each pair; or ranks in snake
    // order.
    auto first_item = [&]() -> int {
        return SNAKE ? item_of_rank((int)blockIdx.x, p) : 2 * (int)blockIdx.x;
    };
    auto next_item = [&](int i, int& step) -> int {
        ++step;
        if constexpr (SNAKE) {
            const int G = (int)gridDim.x;
            return item_of_rank(step * G + ((step & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x), p);
        }
        return (step & 1) ? i + 1 : i - 1 + 2 * (int)gridDim.x;
    };
#ifdef FA_TRACE
    // Loaded once: a trace point is then a clock read and a store.
    unsigned long long* const trace_buf = blockIdx.x < (unsigned)TRACE_CTAS ? g_trace : nullptr;
#endif

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(L::B_QFULL), 1);
        ptx::mbar_init(bar(L::B_QEMPTY), 1);
        for (int s = 0; s < L::KSTAGES; ++s) {
            ptx::mbar_init(bar(L::B_KFULL + s), 1);
            ptx::mbar_init(bar(L::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < L::VSTAGES; ++s) {
            ptx::mbar_init(bar(L::B_VFULL + s), 1);
            ptx::mbar_init(bar(L::B_VEMPTY + s), 1);
        }
        // Softmax-side barriers count warps: each warp arrives once, after __syncwarp.
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(L::B_SFULL + b), 1);
            if constexpr (L::SPLIT) {
                ptx::mbar_init(bar(L::B_PFULL + b), SOFTMAX_WARPS / 2);
                ptx::mbar_init(bar(L::B_PFULL + 2 + b), SOFTMAX_WARPS / 2);
                ptx::mbar_init(bar(L::B_ODONE + b), 1);
            } else {
                ptx::mbar_init(bar(L::B_SREAD + b), SOFTMAX_WARPS);
            }
        }
        if constexpr (!L::SPLIT) {
            ptx::mbar_init(bar(L::B_PFULL), SOFTMAX_WARPS);
            ptx::mbar_init(bar(L::B_ODONE), 1);
        }
        ptx::mbar_init(bar(L::B_OFINAL), 1);
        ptx::mbar_init(bar(L::B_OFREE), EPI_WARPS);
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        ptx::mbar_init(bar(L::B_DRAIN + 1), 1);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(L::B_STFULL + b), SOFTMAX_WARPS);
            ptx::mbar_init(bar(L::B_STFREE + b), EPI_WARPS);
        }
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp < 8) {
        // The ones block of every V stage: bf16 1.0 everywhere (any swizzle).
        const uint32_t one2 = 0x3F803F80u;
        for (int s = 0; s < L::VSTAGES; ++s) {
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
    }
    if (warp == WARP_TMA_V && lane == 0) ptx::prefetch_tensormap(&tm_v);
    if (warp == WARP_MMA_S) {
        ptx::tmem_alloc(sbase + L::OFF_MISC, TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = misc[0];
    // Launched as a programmatic dependent of the kernel before it on the
    // stream: the set-up above overlapped that kernel's last blocks; global
    // memory is touched only after it has completed.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    // Warpgroups 2-3 give up registers that warpgroups 0-1 (the softmax
    // warps) take; each register change heads the code of its warpgroups.
    if (warp >= SOFTMAX_WARPS) {
        ptx::setmaxnreg_dec<L::REGS_OTHER>();
        if (warp == WARP_TMA) {
            // ------------------------------------------- TMA producer: Q and K
            // The whole warp runs the loop (warp-uniform control flow, so the
            // compiler keeps its bookkeeping on the uniform datapath); one elected
            // lane issues each copy: K of every tile as soon as its stage is
            // free, and an item's Q after the item's first K tile, as soon as
            // every score MMA of the item before is done (a K stage frees up
            // a few tiles earlier than Q).  V has a producer of its own
            // (below), so the loads the score stream needs never queue behind
            // a wait for a P.V.
            int gk = 0;
            bool ok = true;
            // Q of item i, the nq-th Q load, once every score MMA of the item
            // before it is done (Q_EMPTY; the phase before cannot alias: this
            // warp waited for it before the load before).
            int nq = 0;
            auto load_q = [&](int i) -> bool {
                if (!warp_wait_bar(bar(L::B_QEMPTY), (uint32_t)(nq & 1) ^ 1u, limit, abort_flag,
                                   0x100 + L::B_QEMPTY))
                    return false;
                const Item iq = item_of<CAUSAL>(i, p);
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(bar(L::B_QFULL), L::Q_BYTES);
                    for (int c = 0; c < L::DBLK; ++c)
                        ptx::tma_load_3d(sbase + L::OFF_Q + c * BLK_BYTES, &tm_q, bar(L::B_QFULL), c * 64, iq.q0,
                                         iq.bh);
                }
                ++nq;
                return true;
            };
            int i = first_item(), step = 0;
            while (ok && i < p.num_items) {
                const Item it = item_of<CAUSAL>(i, p);
                for (int j = 0; ok && j < it.n_kv; ++j) {
                    const int s = gk % L::KSTAGES;
                    const uint32_t ph = (uint32_t)(gk / L::KSTAGES) & 1u;
                    if (!(ok = warp_wait_bar(bar(L::B_KEMPTY + s), ph ^ 1u, limit, abort_flag,
                                             0x100 + L::B_KEMPTY + s)))
                        break;
                    // Test hook: a skipped K tile is never loaded, so the MMA
                    // warp's wait for it runs out (exercises the abort path).
                    const bool skip = gk == p.debug_skip_k && blockIdx.x == 0;
                    if (!skip && ptx::elect_one()) {
                        ptx::mbar_arrive_expect_tx(bar(L::B_KFULL + s), L::KV_BYTES);
                        FA_TRACE_EV(WARP_TMA, gk, 0);
                        for (int c = 0; c < L::DBLK; ++c)
                            ptx::tma_load_3d(sbase + L::OFF_K + s * L::KV_BYTES + c * BLK_BYTES, &tm_k,
                                             bar(L::B_KFULL + s), c * 64, j * BN, it.bh);
                    }
                    ++gk;
                    if (j == 0) {
                        ok = load_q(i);
                        // The next item's Q into L2 now: its load into shared
                        // memory can start only once this item's last score
                        // MMA is done, and would otherwise wait on HBM then.
                        int step_next = step;
                        const int i_next = next_item(i, step_next);
                        if (i_next < p.num_items && ptx::elect_one()) {
                            const Item in = item_of<CAUSAL>(i_next, p);
                            for (int c = 0; c < L::DBLK; ++c) ptx::tma_prefetch_3d(&tm_q, c * 64, in.q0, in.bh);
                        }
                    }
                }
                i = next_item(i, step);
            }
            // Drain: every copy this warp issued must land before exit.
            if (nq > 0) drain_bar(bar(L::B_QFULL), (uint32_t)((nq - 1) & 1), limit, abort_flag, 0x180);
            for (int g = max(0, gk - L::KSTAGES); g < gk; ++g)
                if (!(g == p.debug_skip_k && blockIdx.x == 0))
                    drain_bar(bar(L::B_KFULL + g % L::KSTAGES), (uint32_t)(g / L::KSTAGES) & 1u, limit,
                              abort_flag, 0x181);
        } else if (warp == WARP_TMA_V) {
            // ------------------------------------------------ TMA producer: V
            // V of every tile as soon as its stage is free, i.e. once the P.V
            // that read the stage VSTAGES tiles before is complete.
            int gv = 0;
            bool ok = true;
            for (int i = first_item(), step = 0; ok && i < p.num_items; i = next_item(i, step)) {
                const Item it = item_of<CAUSAL>(i, p);
                for (int j = 0; ok && j < it.n_kv; ++j) {
                    const int s = gv % L::VSTAGES;
                    const uint32_t ph = (uint32_t)(gv / L::VSTAGES) & 1u;
                    if (!(ok = warp_wait_bar(bar(L::B_VEMPTY + s), ph ^ 1u, limit, abort_flag,
                                             0x100 + L::B_VEMPTY + s)))
                        break;
                    if (ptx::elect_one()) {
                        ptx::mbar_arrive_expect_tx(bar(L::B_VFULL + s), L::KV_BYTES);
                        FA_TRACE_EV(WARP_TMA_V, gv, 1);
                        for (int c = 0; c < L::DBLK; ++c)
                            ptx::tma_load_3d(sbase + L::OFF_V + s * L::VSTAGE + c * BLK_BYTES, &tm_v,
                                             bar(L::B_VFULL + s), c * 64, j * BN, it.bh);
                    }
                    ++gv;
                }
            }
            // Drain: every copy this warp issued must land before exit.
            for (int g = max(0, gv - L::VSTAGES); g < gv; ++g)
                drain_bar(bar(L::B_VFULL + g % L::VSTAGES), (uint32_t)(g / L::VSTAGES) & 1u, limit,
                          abort_flag, 0x182);
        } else if (warp == WARP_MMA_S) {
            // ------------------------------------------------- score MMA issuer
            // S for global tile g = Q K_j^T into S buffer g & 1; K-major operands,
            // 16 columns per MMA.  Descriptors are built once; stepping through K
            // only moves the start-address field (bits 0-13, in 16-byte units).
            constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(BM, BN, false);
            const uint64_t q_desc = ptx::sdesc_sw128(sbase + L::OFF_Q, 16, 1024);
            const uint64_t k_desc0 = ptx::sdesc_sw128(sbase + L::OFF_K, 16, 1024);
            //
            // This warp also tells the softmax warps that S of a tile is complete:
            // it waits on the MMA completion (an mbarrier) long before they need
            // it and arrives on a named barrier, which they meet in a few cycles.
            // An mbarrier poll of theirs would queue in shared memory behind the
            // score MMAs' operand reads (hundreds of cycles on every tile).  S of
            // tile g - 1 is signalled before the waits for tile g, so a new item's
            // Q load never delays the last tile of the previous item.  The loops
            // walk every item and tile also after an abort (the MMAs are skipped),
            // so that every S-ready generation is signalled.
            int g = 0, k = 0;  // tiles and items done
            bool ok = true;
            auto signal_s_ready = [&](int gg) {
                if (ok) ok = warp_wait_bar(bar(L::B_SFULL + (gg & 1)), (uint32_t)(gg >> 1) & 1u, limit, abort_flag,
                                           0x200 + L::B_SFULL + (gg & 1));
                ptx::tc_fence_before_sync();
                __syncwarp();
                if constexpr (L::SPLIT) {
                    nb_signal(NB_SREADY_SPLIT0 + (uint32_t)(gg % 3), NB_SREADY_SPLIT_COUNT, ok);       // half 0
                    nb_signal(NB_SREADY_SPLIT0 + 3u + (uint32_t)(gg % 3), NB_SREADY_SPLIT_COUNT, ok);  // half 1
                } else {
                    nb_signal(NB_SREADY0 + (uint32_t)(gg % 3), NB_SREADY_COUNT, ok);
                }
            };
            for (int i = first_item(), step = 0; i < p.num_items; i = next_item(i, step), ++k) {
                const int n = item_of<CAUSAL>(i, p).n_kv;
                for (int j = 0; j < n; ++j, ++g) {
                    const int b = g & 1;
                    const int s = g % L::KSTAGES;
                    if (g >= 1) signal_s_ready(g - 1);
                    if (j == 0 && ok)
                        ok = warp_wait_bar(bar(L::B_QFULL), (uint32_t)(k & 1), limit, abort_flag, 0x200 + L::B_QFULL);
                    // K of tile g was loaded long before: its check goes first, the
                    // wait for the softmax warps' signal last.
                    if (ok) ok = warp_wait_bar(bar(L::B_KFULL + s), (uint32_t)(g / L::KSTAGES) & 1u, limit, abort_flag,
                                               0x200 + L::B_KFULL + s);
                    // Buffer b is free once every softmax warp has read S of tile
                    // g - 2 (the phase before cannot alias: S of g - 2 was issued
                    // only after S of g - 4 had been read).
                    // Split design: P of tile g - 2 lies over its scores, so buffer
                    // b is free once both halves' P.V of g - 2 are complete.
                    if (g >= 2 && ok) {
                        const int bb = L::SPLIT ? L::B_ODONE + b : L::B_SREAD + b;
                        ok = warp_wait_bar(bar(bb), (uint32_t)((g - 2) >> 1) & 1u, limit, abort_flag, 0x200 + bb);
                    }
                    if (!ok) continue;
                    if (lane == 0) FA_TRACE_EV(WARP_MMA_S, g, 0);
                    ptx::tc_fence_after_sync();
                    const uint32_t d_tmem = tmem + (b ? TM_S1 : TM_S0);
                    const uint64_t k_desc = k_desc0 + (uint64_t)((s * L::KV_BYTES) >> 4);
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = ((uint32_t)(kk >> 2) * BLK_BYTES + (uint32_t)(kk & 3) * 32) >> 4;
                        if (ptx::elect_one())
                            ptx::mma_ss(d_tmem, q_desc + koff, k_desc + koff, IDESC_S, kk > 0 ? 1u : 0u);
                    }
                    if (ptx::elect_one()) {
                        ptx::tc_commit(bar(L::B_KEMPTY + s));
                        ptx::tc_commit(bar(L::B_SFULL + b));
                        // Q may be replaced once the item's last score MMA is done.
                        if (j == n - 1) ptx::tc_commit(bar(L::B_QEMPTY));
                        FA_TRACE_EV(WARP_MMA_S, g, 1);
                    }
                }
            }
            if (g >= 1) signal_s_ready(g - 1);
            // Drain: all MMAs issued by this warp complete before TMEM is freed.
            if (ptx::elect_one()) ptx::tc_commit(bar(L::B_DRAIN));
            drain_bar(bar(L::B_DRAIN), 0, limit, abort_flag, 0x280);
        } else if (warp == WARP_MMA_O) {
            // ------------------------------------------------- P.V MMA issuer
            // [O | l~] (+)= P [V | 1] for global tile g: A = P from TMEM (2 bf16
            // per column, 8 columns per 16 keys); B MN-major (value columns
            // contiguous): 64-column blocks BLK_BYTES apart (the ones block follows
            // the value blocks), 8-key groups 1024 bytes apart.
            if constexpr (L::SPLIT) {
                // [O_h | l~_h] (+)= P_h [V_h | 1] for global tile g and each half h:
                // A = P_h from TMEM (over the half's scores in S buffer g & 1; 2 bf16
                // per column, 8 columns per 16 keys), B = value rows 64h .. 64h+63,
                // MN-major (value columns contiguous): 64-column blocks BLK_BYTES
                // apart (the ones block follows the value blocks), 8-key groups 1024
                // bytes apart.  Each half's P is taken as soon as it is written.
                constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(BM, D + 16, true);
                const uint64_t v_desc0 = ptx::sdesc_sw128(sbase + L::OFF_V, BLK_BYTES, 1024);
                int g = 0, k = 0;  // tiles and items done
                bool ok = true;
                for (int i = first_item(), step = 0; ok && i < p.num_items; i = next_item(i, step), ++k) {
                    const int n = item_of<CAUSAL>(i, p).n_kv;
                    // The first P.V of an item overwrites O: wait until the softmax
                    // warps have read out the previous item's O.
                    if (!(ok = warp_wait_bar(bar(L::B_OFREE), (uint32_t)(k & 1) ^ 1u, limit, abort_flag,
                                             0x200 + L::B_OFREE)))
                        break;
                    for (int j = 0; ok && j < n; ++j, ++g) {
                        const int s = g % L::VSTAGES;
                        const int b = g & 1;
                        // V of tile g, loaded long before, is checked first: an mbarrier
                        // check is slow while the score MMAs stream their operands, and
                        // it then overlaps the softmax warps' work on P.
                        if (!(ok = warp_wait_bar(bar(L::B_VFULL + s), (uint32_t)(g / L::VSTAGES) & 1u, limit,
                                                 abort_flag, 0x200 + L::B_VFULL + s)))
                            break;
                        if (lane == 0) FA_TRACE_EV(WARP_MMA_O, g, 3);
                        const uint64_t v_desc = v_desc0 + (uint64_t)((s * L::VSTAGE) >> 4);
                        const uint32_t s_tm = tmem + (b ? TM_S1 : TM_S0);
    #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // P_h of tile g (per S buffer: the phase before, tile g - 2,
                            // was consumed by this warp, so parity cannot alias).
                            if (!(ok = warp_wait_bar(bar(L::B_PFULL + 2 * h + b), (uint32_t)(g >> 1) & 1u, limit,
                                                     abort_flag, 0x200 + L::B_PFULL + 2 * h + b)))
                                break;
                            ptx::tc_fence_after_sync();
    #pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                if (ptx::elect_one())
                                    ptx::mma_ts(tmem + TM_O + (uint32_t)h * L::O_STRIDE, s_tm + (uint32_t)(h * 64 + kk * 8),
                                                v_desc + (uint64_t)(((h * 64 + kk * 16) * 128) >> 4), IDESC_O,
                                                (j > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        if (!ok) break;
                        if (ptx::elect_one()) {
                            // The commits cover every MMA this warp issued so far.
                            ptx::tc_commit(bar(L::B_VEMPTY + s));
                            ptx::tc_commit(bar(L::B_ODONE + b));
                            if (j == n - 1) ptx::tc_commit(bar(L::B_OFINAL));
                            FA_TRACE_EV(WARP_MMA_O, g, 4);
                        }
                    }
                }
            } else {
                constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(BM, D + 16, true);
                const uint64_t v_desc0 = ptx::sdesc_sw128(sbase + L::OFF_V, BLK_BYTES, 1024);
                const uint32_t p_tmem = tmem + TM_P;
                int g = 0, k = 0;  // tiles and items done
                bool ok = true;
                for (int i = first_item(), step = 0; ok && i < p.num_items; i = next_item(i, step), ++k) {
                    const int n = item_of<CAUSAL>(i, p).n_kv;
                    // The first P.V of an item overwrites O: wait until the softmax
                    // warps have read out the previous item's O.
                    if (!(ok = warp_wait_bar(bar(L::B_OFREE), (uint32_t)(k & 1) ^ 1u, limit, abort_flag,
                                             0x200 + L::B_OFREE)))
                        break;
                    for (int j = 0; j < n; ++j, ++g) {
                        const int s = g % L::VSTAGES;
                        // V of tile g, loaded long before, is checked first: an mbarrier
                        // check is slow while the score MMAs stream their operands, and
                        // it then overlaps the softmax warps' work on P.  Then P of tile
                        // g (the phase before is P of g - 1, which this warp has
                        // consumed, so parity cannot alias).
                        if (!(ok = warp_wait_bar(bar(L::B_VFULL + s), (uint32_t)(g / L::VSTAGES) & 1u, limit,
                                                 abort_flag, 0x200 + L::B_VFULL + s)))
                            break;
                        if (lane == 0) FA_TRACE_EV(WARP_MMA_O, g, 3);
                        if (!(ok = warp_wait_bar(bar(L::B_PFULL), (uint32_t)(g & 1), limit, abort_flag,
                                                 0x200 + L::B_PFULL)))
                            break;
                        if (lane == 0) FA_TRACE_EV(WARP_MMA_O, g, 2);
                        ptx::tc_fence_after_sync();
                        const uint64_t v_desc = v_desc0 + (uint64_t)((s * L::VSTAGE) >> 4);
    #pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            if (ptx::elect_one())
                                ptx::mma_ts(tmem + TM_O, p_tmem + (uint32_t)kk * 8,
                                            v_desc + (uint64_t)(kk * ((16 * 128) >> 4)), IDESC_O,
                                            (j > 0 || kk > 0) ? 1u : 0u);
                            if (kk == 0 && lane == 0) FA_TRACE_EV(WARP_MMA_O, g, 5);
                            if (kk == 7 && lane == 0) FA_TRACE_EV(WARP_MMA_O, g, 7);
                        }
                        if (ptx::elect_one()) {
                            ptx::tc_commit(bar(L::B_VEMPTY + s));
                            ptx::tc_commit(bar(L::B_ODONE));
                            if (j == n - 1) ptx::tc_commit(bar(L::B_OFINAL));
                            FA_TRACE_EV(WARP_MMA_O, g, 4);
                        }
                    }
                }
            }
            if (ptx::elect_one()) ptx::tc_commit(bar(L::B_DRAIN + 1));
            drain_bar(bar(L::B_DRAIN + 1), 0, limit, abort_flag, 0x281);
        } else if (warp < WARP_EPI0 + EPI_WARPS) {
            // ------------------------------------------------------ epilogue warps
            // Warp 8 + q serves TMEM lane quarter q: query rows 32q .. 32q+31 of
            // every item, one row a thread.  Per item: the statistics the softmax
            // warps left in TMEM (slot item & 1), then, once the item's last P.V
            // is complete, O and l~:
            //   D = 128: out = O / l~,  lse = (m + log2(l_0 + l_1)) ln 2 (both
            //     halves of a row share the reference max m);
            //   split design (D = 64): with w_h = 2^(m_h - M), M = max(m_0, m_1),
            //     out = (w_0 O_0 + w_1 O_1) / (w_0 l~_0 + w_1 l~_1),
            //     lse = (M + log2(w_0 l_0 + w_1 l_1)) ln 2,
            //   the merge of two split-key partial results; O stays an exact
            //   convex combination of value rows.
            // O_FREE is arrived once O has been read, without release semantics
            // (nothing waits for the stores); a head size d below D was
            // zero-padded by the TMA loads, so the padded columns are not stored.
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;  // query row in the item == TMEM lane
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const int ostride = PAD ? p.d : D;
            bool ok = true;
            int kitem = 0;
            for (int i = first_item(), step = 0; ok && i < p.num_items; i = next_item(i, step), ++kitem) {
                const Item it = item_of<CAUSAL>(i, p);
                const int slot = kitem & 1;
                if (!(ok = warp_wait_bar(bar(L::B_STFULL + slot), (uint32_t)(kitem >> 1) & 1u, limit, abort_flag,
                                         0x480 + L::B_STFULL + slot)))
                    break;
                ptx::tc_fence_after_sync();
                uint32_t st[4];  // m_0, m_1, l_0, l_1
                ptx::tmem_ld4(tmem + lane_off + TM_ST + 4u * (uint32_t)slot, st);
                ptx::tmem_wait_ld_only();
                ptx::reg_fence4(st);
                ptx::tc_fence_before_sync();
                __syncwarp();
                // The slot may be written again (the split design waits for
                // this; at D = 128 the slot's reuse is ordered through O_FREE).
                if (L::SPLIT && lane == 0) ptx::mbar_arrive_relaxed(bar(L::B_STFREE + slot));
                // The item's last P.V (the phase before, the previous item's, was
                // waited for here before O_FREE let this item's first P.V start).
                if (!(ok = warp_wait_bar(bar(L::B_OFINAL), (uint32_t)(kitem & 1), limit, abort_flag,
                                         0x480 + L::B_OFINAL)))
                    break;
                ptx::tc_fence_after_sync();
                const int q_idx = it.q0 + row;
                const bool row_ok = q_idx < N;
                __nv_bfloat16* const orow = p.o + ((int64_t)it.bh * N + q_idx) * ostride;
                const uint32_t o0 = tmem + lane_off + TM_O;
                float m, l;
                if constexpr (L::SPLIT) {
                    const float m0 = __uint_as_float(st[0]), m1 = __uint_as_float(st[1]);
                    m = fmaxf(m0, m1);
                    const float w0 = ptx::ex2(m0 - m), w1 = ptx::ex2(m1 - m);
                    l = __uint_as_float(st[2]) * w0 + __uint_as_float(st[3]) * w1;
                    const uint32_t o1 = o0 + L::O_STRIDE;
                    const float lr0 = __uint_as_float(ptx::tmem_ld1_wait(o0 + D));
                    const float lr1 = __uint_as_float(ptx::tmem_ld1_wait(o1 + D));
                    const float inv = 1.0f / (lr0 * w0 + lr1 * w1);
                    const float c0 = w0 * inv, c1 = w1 * inv;
                        if constexpr (!PAD) {
                        uint32_t w[32];  // the row: D = 64 columns
#pragma unroll
                        for (int ch = 0; ch < D / 16; ++ch) {
                            uint32_t oa[16], ob[16];
                            ptx::tmem_ld16(o0 + ch * 16, oa);
                            ptx::tmem_ld16(o1 + ch * 16, ob);
                            ptx::tmem_wait_ld_only();
                            ptx::reg_fence16(oa);
                            ptx::reg_fence16(ob);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                w[8 * ch + c] = ptx::pack_bf16x2(
                                    fmaf(__uint_as_float(oa[2 * c]), c0, __uint_as_float(ob[2 * c]) * c1),
                                    fmaf(__uint_as_float(oa[2 * c + 1]), c0, __uint_as_float(ob[2 * c + 1]) * c1));
                        }
                        // The whole row is in registers (the loads above have
                        // completed): O is released to the next item's first P.V
                        // before the stores.
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_relaxed(bar(L::B_OFREE));
                        const int row0 = it.q0 + quarter * 32;
                        store_rows_coalesced(w, p.o + ((int64_t)it.bh * N + row0) * D, lane, N - row0, D);
                    } else {
    #pragma unroll
                        for (int ch = 0; ch < D / 16; ++ch) {
                            uint32_t oa[16], ob[16];
                            ptx::tmem_ld16(o0 + ch * 16, oa);
                            ptx::tmem_ld16(o1 + ch * 16, ob);
                            ptx::tmem_wait_ld_only();
                            ptx::reg_fence16(oa);
                            ptx::reg_fence16(ob);
                            uint32_t w[8];
        #pragma unroll
                            for (int c = 0; c < 8; ++c)
                                w[c] = ptx::pack_bf16x2(
                                    fmaf(__uint_as_float(oa[2 * c]), c0, __uint_as_float(ob[2 * c]) * c1),
                                    fmaf(__uint_as_float(oa[2 * c + 1]), c0, __uint_as_float(ob[2 * c + 1]) * c1));
                            if (row_ok) {
        #pragma unroll
                                for (int u = 0; u < 2; ++u)
                                    if (!PAD || ch * 16 + u * 8 < p.d)
                                        ptx::st_global_v4(orow + ch * 16 + u * 8, w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                          w[4 * u + 3]);
                            }
                        }
                    }
                } else {
                    m = __uint_as_float(st[0]);
                    l = __uint_as_float(st[2]) + __uint_as_float(st[3]);
                    const float inv = 1.0f / __uint_as_float(ptx::tmem_ld1_wait(o0 + D));  // l~
                        if constexpr (!PAD) {
                        const int row0 = it.q0 + quarter * 32;
#pragma unroll
                        for (int hh = 0; hh < D / 64; ++hh) {
                            uint32_t w[32];  // 64 columns of the row
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch) {
                                uint32_t o[16];
                                ptx::tmem_ld16(o0 + hh * 64 + ch * 16, o);
                                ptx::tmem_wait_ld_only();
                                ptx::reg_fence16(o);
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    w[8 * ch + c] = ptx::pack_bf16x2(__uint_as_float(o[2 * c]) * inv,
                                                                     __uint_as_float(o[2 * c + 1]) * inv);
                            }
                            store_rows_coalesced(w, p.o + ((int64_t)it.bh * N + row0) * D + hh * 64, lane, N - row0, D);
                        }
                    } else {
    #pragma unroll
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t o[32];
                            ptx::tmem_ld32(o0 + ch * 32, o);
                            ptx::tmem_wait_ld(o);
                            uint32_t w[16];
        #pragma unroll
                            for (int c = 0; c < 16; ++c)
                                w[c] = ptx::pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
                            if (row_ok) {
        #pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    if (!PAD || ch * 32 + u * 8 < p.d)
                                        ptx::st_global_v4(orow + ch * 32 + u * 8, w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                          w[4 * u + 3]);
                            }
                        }
                    }
                }
                // O has been read (every load above has completed): the next
                // item's first P.V may overwrite it.  (The split design's
                // unpadded path released it before its stores.  At D = 128 the
                // stores come first: released earlier, they ran beside the next
                // item's MMAs and slowed them more than the wait costs.)
                if constexpr (!(L::SPLIT && !PAD)) {
                    ptx::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_relaxed(bar(L::B_OFREE));
                }
                if (row_ok) p.lse[(int64_t)it.bh * N + q_idx] = (m + ptx::lg2(l)) * 0.69314718055994530942f;
            }
        }
    } else {
        ptx::setmaxnreg_inc<L::REGS_SOFTMAX>();
            if constexpr (L::SPLIT) {
                // ------------------------------------- softmax warps, split design
                // Warp w serves query rows 32*(w%4) .. +31 (its TMEM lane quarter) and
                // score columns 64*h .. +63, h = w/4, with a state of its own: its
                // reference max, its row sum, its P (written over its half of the S
                // buffer) and its accumulator [O_h | l~_h] = sum over tiles of
                // P_h [V_h | 1].  The two halves of a row meet once per item, in the
                // epilogue.
                const int quarter = warp & 3;
                const int half = warp >> 2;
                const int row = quarter * 32 + lane;      // query row in the item == TMEM lane
                const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
                const uint32_t o_mine = tmem + lane_off + TM_O + (uint32_t)half * L::O_STRIDE;
                const float sl2 = p.scale_log2;
                const uint32_t nb_sready = NB_SREADY_SPLIT0 + 3u * (uint32_t)half;
                bool ok = true;
                int g = 0;      // tiles done
                int kitem = 0;  // items done

                for (int i = first_item(), step = 0; i < p.num_items; i = next_item(i, step)) {
                    const Item it = item_of<CAUSAL>(i, p);
                    const int q_idx = it.q0 + row;
                    const int key_max = CAUSAL ? min(q_idx, N - 1) : N - 1;
                    const int cta_key_max = CAUSAL ? min(it.q0, N - 1) : N - 1;  // smallest key_max of the item
                    float m_ref = -INFINITY;
                    // This half-row's sum of probabilities, as four packed fp32 pairs.
                    uint64_t lsum[4] = {0ull, 0ull, 0ull, 0ull};
                    {
                    // This half-row's scores (fp32 bit patterns), used in place: the
                    // packed fp32x2 arithmetic takes neighbouring load registers as
                    // its operand pairs.
                    uint32_t sr[64];

                    for (int j = 0; j < it.n_kv; ++j, ++g) {
                        const int b = g & 1;
                        const uint32_t s_half = tmem + lane_off + (b ? TM_S1 : TM_S0) + (uint32_t)half * 64;
                        // S of tile g is in TMEM (met on every tile, also after an abort).
                        ptx::named_barrier_sync(nb_sready + (uint32_t)(g % 3), NB_SREADY_SPLIT_COUNT);
                        if (!ok) continue;
                        ptx::tc_fence_after_sync();
                        // The load also returns the max of the 64 scores (the TMEM
                        // load's reduction); a masked tile takes it again after the
                        // mask.
                        float red;
                        ptx::tmem_ld64_max(s_half, sr, red);
                        if (lane == 0) FA_TRACE_EV(warp, g, 0);
                        ptx::tmem_wait_ld64_max(sr, red);
                        if (lane == 0) FA_TRACE_EV(warp, g, 1);
                        // Causal diagonal tile / keys past N: -inf before the max.
                        const int k0 = j * BN + half * 64;
                        if (j * BN + BN - 1 > cta_key_max) {
    #pragma unroll
                            for (int c = 0; c < 64; ++c)
                                if (k0 + c > key_max) sr[c] = __float_as_uint(-INFINITY);
                            red = max64(sr);
                        }
                        const float m_tile = red * sl2;  // scale > 0, so max commutes with it
                        if (lane == 0) FA_TRACE_EV(warp, g, 2);

                        // A half-row may have no visible key yet (its reference then
                        // stays -inf and its P, O_h and l are 0).
                        if (j == 0) {
                            m_ref = m_tile;
                        } else {
                            const float m_new = fmaxf(m_ref, m_tile);
                            const bool need = m_new > m_ref + RESCALE_LOG2;
                            if (__any_sync(0xffffffffu, need)) {
                                // O_h holds everything up to the previous tile once
                                // both halves' P.V of it are done (the phase before,
                                // tile g - 3, cannot alias: tile g - 1 was issued only
                                // after it).
                                if (!(ok = warp_wait_bar(bar(L::B_ODONE + ((g - 1) & 1)), (uint32_t)((g - 1) >> 1) & 1u,
                                                         limit, abort_flag, 0x300 + L::B_ODONE + ((g - 1) & 1))))
                                    continue;
                                ptx::tc_fence_after_sync();
                                const float corr = ptx::ex2(m_ref - m_new);
    #pragma unroll
                                for (int c = 0; c < 4; ++c) lsum[c] = ptx::f2_mul(lsum[c], ptx::f2_pack(corr, corr));

                                m_ref = m_new;
                                scale_row<D>(o_mine, corr);
                                uint32_t lt[8];
                                ptx::tmem_ld8(o_mine + D, lt);
                                ptx::tmem_wait_ld_only();
                                ptx::reg_fence8(lt);
    #pragma unroll
                                for (int c = 0; c < 8; ++c) lt[c] = __float_as_uint(__uint_as_float(lt[c]) * corr);
                                ptx::tmem_st8(o_mine + D, lt);
                                ptx::tmem_wait_st();
                            }
                        }

                        // P = 2^(s*c - m_ref), rounded to bf16 for the P.V MMA.  The
                        // scaling and the sums use packed fp32x2 instructions: fewer
                        // issue slots, which the MMA issuers on the same sub-partitions
                        // need.
                        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
                        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                        const uint64_t neg_m2 = ptx::f2_pack(-m_use, -m_use);
                        uint32_t pk[32];
    #pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            float x0, x1;
                            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])),
                                                       sl2x2, neg_m2),
                                           x0, x1);
                            const float a0 = ptx::ex2(x0);
                            const float a1 = ptx::ex2(x1);
                            lsum[c & 3] = ptx::f2_add(lsum[c & 3], ptx::f2_pack(a0, a1));
                            pk[c] = ptx::pack_bf16x2(a0, a1);
                        }
                        if (lane == 0) FA_TRACE_EV(warp, g, 3);

                        // P over this half's scores (read into registers above).
                        ptx::tmem_st32(s_half, pk);
                        ptx::tmem_wait_st();
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(L::B_PFULL + 2 * half + b));
                        if (lane == 0) FA_TRACE_EV(warp, g, 5);
                    }
                    }

                    // ------------------------------- the item to the epilogue warps
                    // This half-row's reference max and fp32 row sum go to the
                    // item's statistics slot in TMEM (item parity; columns m_0, m_1,
                    // l_0, l_1) once the epilogue warps have read what the slot held
                    // two items ago; one arrival per warp says it is written.  The
                    // softmax warps then start the next item at once.
                    {
                        float l_lo, l_hi;
                        ptx::f2_unpack(ptx::f2_add(ptx::f2_add(lsum[0], lsum[1]), ptx::f2_add(lsum[2], lsum[3])), l_lo,
                                       l_hi);
                        const int slot = kitem & 1;
                        if (ok)
                            ok = warp_wait_bar(bar(L::B_STFREE + slot), ((uint32_t)(kitem >> 1) & 1u) ^ 1u, limit,
                                               abort_flag, 0x380 + L::B_STFREE + slot);
                        if (ok) {
                            const uint32_t st = tmem + lane_off + TM_ST + 4u * (uint32_t)slot;
                            ptx::tmem_st1(st + (uint32_t)half, __float_as_uint(m_ref));
                            ptx::tmem_st1(st + 2u + (uint32_t)half, __float_as_uint(l_lo + l_hi));
                            ptx::tmem_wait_st();
                            ptx::tc_fence_before_sync();
                        }
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(L::B_STFULL + slot));
                        ++kitem;
                    }
                }
            } else {
                // ---------------------------------------------------- softmax warps
                const int quarter = warp & 3;
                const int half = warp >> 2;               // score columns [64*half, 64*half+64)
                const int row = quarter * 32 + lane;      // query row in the item == TMEM lane
                const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
                const uint32_t o_cols = tmem + lane_off + TM_O + (uint32_t)half * (D / 2);
                const uint32_t l_cols = tmem + lane_off + L::TM_L + (uint32_t)half * 8;
                const float sl2 = p.scale_log2;
                bool ok = true;
                int g = 0;      // tiles done
                int kitem = 0;  // items done

                // Every softmax warp runs the same items and tiles and reaches each
                // named barrier the same number of times, also after an abort
                // (ok == false: the work is skipped, the barriers are not), so a named
                // barrier never waits for a warp that has left the loop.
                for (int i = first_item(), step = 0; i < p.num_items; i = next_item(i, step)) {
                    const Item it = item_of<CAUSAL>(i, p);
                    const int q_idx = it.q0 + row;
                    const int key_max = CAUSAL ? min(q_idx, N - 1) : N - 1;
                    const int cta_key_max = CAUSAL ? min(it.q0, N - 1) : N - 1;  // smallest key_max of the item
                    float m_ref = -INFINITY;
                    // This half-row's sum of probabilities, as four packed fp32 pairs.
                    uint64_t lsum[4] = {0ull, 0ull, 0ull, 0ull};
                    {
                    // This half-row's scores (fp32 bit patterns), used in place: the
                    // packed fp32x2 arithmetic takes neighbouring load registers as
                    // its operand pairs.
                    uint32_t sr[64];

                    for (int j = 0; j < it.n_kv; ++j, ++g) {
                        const int b = g & 1;
                        // S of tile g is in TMEM (met on every tile, also after an abort).
                        ptx::named_barrier_sync(NB_SREADY0 + (uint32_t)(g % 3), NB_SREADY_COUNT);
                        // The load also returns the max of the 64 scores (the TMEM
                        // load's reduction); a masked tile takes it again after the
                        // mask.
                        float red = -INFINITY;
                        if (ok) {
                            ptx::tc_fence_after_sync();
                            ptx::tmem_ld64_max(tmem + lane_off + (b ? TM_S1 : TM_S0) + (uint32_t)half * 64, sr, red);
                        }
                        if (lane == 0) FA_TRACE_EV(warp, g, 0);
                        float mx = -INFINITY;
                        if (ok) {
                            ptx::tmem_wait_ld64_max(sr, red);
                            // The scores are in registers: S of tile g + 2 may now be
                            // written into this buffer.
                            ptx::tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive(bar(L::B_SREAD + b));
                            if (lane == 0) FA_TRACE_EV(warp, g, 1);
                            // Causal diagonal tile / keys past N: -inf before the max.
                            const int k0 = j * BN + half * 64;
                            if (j * BN + BN - 1 > cta_key_max) {
    #pragma unroll
                                for (int c = 0; c < 64; ++c)
                                    if (k0 + c > key_max) sr[c] = __float_as_uint(-INFINITY);
                                mx = max64(sr);
                            } else {
                                mx = red;
                            }
                            ptx::tmem_st1(tmem + lane_off + TM_MX + (uint32_t)(b * 2 + half), __float_as_uint(mx));
                            ptx::tmem_wait_st();
                            ptx::tc_fence_before_sync();
                        }
                        // Row max: this half's, then the partner warp's through two TMEM
                        // columns per S buffer (TMEM, unlike shared memory, does not
                        // queue behind the score MMAs' operand reads).  The slot is
                        // rewritten two tiles later, after the partner has passed the
                        // next tile's barrier, so after it read this value.
                        ptx::named_barrier_sync(NB_PAIR0 + quarter, 64);
                        if (lane == 0) FA_TRACE_EV(warp, g, 2);
                        if (!ok) continue;
                        ptx::tc_fence_after_sync();
                        const uint32_t mx_other = tmem + lane_off + TM_MX + (uint32_t)(b * 2 + (half ^ 1));
                        mx = fmaxf(mx, __uint_as_float(ptx::tmem_ld1_wait(mx_other)));
                        const float m_tile = mx * sl2;  // scale > 0, so max commutes with it

                        // [O | l~] and the P buffer are free of tile g - 1 once its P.V
                        // is done (O_DONE; the phase before, P.V of g - 2, was waited
                        // for before P of g - 1 was written, so parity cannot alias).
                        bool o_done = g == 0;
                        auto wait_o_done = [&]() -> bool {
                            if (o_done) return true;
                            if (!warp_wait_bar(bar(L::B_ODONE), (uint32_t)(g - 1) & 1u, limit, abort_flag,
                                               0x300 + L::B_ODONE))
                                return false;
                            ptx::tc_fence_after_sync();
                            o_done = true;
                            return true;
                        };
                        if (j == 0) {
                            m_ref = (m_tile == -INFINITY) ? 0.f : m_tile;
                        } else {
                            const float m_new = fmaxf(m_ref, m_tile);
                            const bool need = m_new > m_ref + RESCALE_LOG2;
                            // Both halves of a row see the same values, so they decide alike.
                            if (__any_sync(0xffffffffu, need)) {
                                // [O | l~] hold everything up to the previous tile once
                                // its P.V is done.
                                if (!(ok = wait_o_done())) continue;
                                const float corr = ptx::ex2(m_ref - m_new);
    #pragma unroll
                                for (int c = 0; c < 4; ++c) lsum[c] = ptx::f2_mul(lsum[c], ptx::f2_pack(corr, corr));
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

                        // P = 2^(s*c - m_ref), rounded to bf16 for the P.V MMA.  The
                        // scaling and the sums use packed fp32x2 instructions: fewer
                        // issue slots, which the MMA issuer on the same sub-partition
                        // needs.
                        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
                        const uint64_t neg_m2 = ptx::f2_pack(-m_ref, -m_ref);
                        uint32_t pk[32];
    #pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            float x0, x1;
                            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])),
                                                       sl2x2, neg_m2),
                                           x0, x1);
                            const float a0 = ptx::ex2(x0);
                            const float a1 = ptx::ex2(x1);
                            lsum[c & 3] = ptx::f2_add(lsum[c & 3], ptx::f2_pack(a0, a1));
                            pk[c] = ptx::pack_bf16x2(a0, a1);
                        }
                        if (lane == 0) FA_TRACE_EV(warp, g, 3);

                        // P into the P buffer once the previous tile's P.V has read it.
                        if (!(ok = wait_o_done())) continue;
                        ptx::tmem_st32(tmem + lane_off + TM_P + (uint32_t)half * 32, pk);
                        ptx::tmem_wait_st();
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(L::B_PFULL));
                        if (lane == 0) FA_TRACE_EV(warp, g, 5);
                    }
                    }

                    // ------------------------------- the item to the epilogue warps
                    // This half-row's reference max and fp32 row sum go to the
                    // item's statistics slot in TMEM (item parity; columns m_0, m_1,
                    // l_0, l_1) once the epilogue warps have read what the slot held
                    // two items ago; one arrival per warp says it is written.  The
                    // softmax warps then start the next item at once.
                    {
                        float l_lo, l_hi;
                        ptx::f2_unpack(ptx::f2_add(ptx::f2_add(lsum[0], lsum[1]), ptx::f2_add(lsum[2], lsum[3])), l_lo,
                                       l_hi);
                        // The slot held item kitem - 2, and its statistics have
                        // been read: they were read before O_FREE of that item,
                        // which the first P.V of item kitem - 1 waited for, and
                        // every P of this item was written after a P.V of item
                        // kitem - 1 or later was complete (O_DONE).
                        const int slot = kitem & 1;
                        if (ok) {
                            const uint32_t st = tmem + lane_off + TM_ST + 4u * (uint32_t)slot;
                            ptx::tmem_st1(st + (uint32_t)half, __float_as_uint(m_ref));
                            ptx::tmem_st1(st + 2u + (uint32_t)half, __float_as_uint(l_lo + l_hi));
                            ptx::tmem_wait_st();
                            ptx::tc_fence_before_sync();
                        }
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(L::B_STFULL + slot));
                        ++kitem;
                    }
                }
            }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA_S) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace fa
