// C ABI of the attention-forward library: argument checks, TMA descriptors,
// kernel selection and launch.  Declarations and the contract: include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <utility>

#include "fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_decode_kernel.cuh"
#include "fa_ew_kernel.cuh"
#include "fa_fwd_kernel.cuh"

namespace {

constexpr int FA_VERSION = 100;  // 0.1.0
constexpr uint64_t DEFAULT_WAIT_LIMIT_NS = 1000000000ull;
constexpr int MAX_DEVICES = 64;

std::atomic<uint64_t> g_wait_limit_ns{DEFAULT_WAIT_LIMIT_NS};
std::atomic<int> g_debug_skip_k{-1};
std::atomic<int> g_debug_schedule{-1};  // causal item order: -1 by size, 0 pairs, 1 cost order

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// (B*H, N, d) bf16 viewed as a 3-D tensor (d innermost); box = 64 columns x
// `rows` rows x 1 head, 128-byte swizzle.  Rows past N read as zero on loads
// and are dropped on stores.
bool make_map(CUtensorMap* map, const void* base, int64_t BH, int64_t N, int64_t d, uint32_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)(N * d * 2)};
    cuuint32_t box[3] = {64, rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// make_map through a small per-thread cache of recent encodes.  The encode is
// a pure function of its arguments (address, sizes, box rows; the data type,
// swizzle and fill are fixed), so a hit returns exactly the map a fresh
// encode would.  Repeated calls on the same buffers then skip the driver's
// encode (three per forward call).
bool cached_map(CUtensorMap* map, const void* base, int64_t BH, int64_t N, int64_t d, uint32_t rows)
{
    struct Entry {
        CUtensorMap map;
        const void* base;
        int64_t BH, N, d;
        uint32_t rows;
        bool valid;
    };
    constexpr int SLOTS = 8;
    thread_local Entry cache[SLOTS] = {};
    thread_local unsigned next = 0;
    for (int i = 0; i < SLOTS; ++i) {
        const Entry& e = cache[i];
        if (e.valid && e.base == base && e.BH == BH && e.N == N && e.d == d && e.rows == rows) {
            *map = e.map;
            return true;
        }
    }
    if (!make_map(map, base, BH, N, d, rows)) return false;
    Entry& e = cache[next++ % SLOTS];
    e.map = *map;
    e.base = base;
    e.BH = BH;
    e.N = N;
    e.d = d;
    e.rows = rows;
    e.valid = true;
    return true;
}

// The backward's fp32 dQ accumulator (B*H, Np, d) as a 3-D tensor; box = 32
// columns x 64 rows x 1 head, no swizzle (the reduce-add source is a plain
// row-major 64 x 32 block).
bool make_acc_map(CUtensorMap* map, void* base, int64_t BH, int64_t Np, int64_t d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Np, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)(d * 4), (cuuint64_t)(Np * d * 4)};
    cuuint32_t box[3] = {32, (cuuint32_t)fa::bwd::BQ, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head sizes the forward and backward take: multiples of 8 up to 128.  They
// run in the kernel instance for 64 (d <= 64) or 128 columns; the TMA loads
// fill the columns past d with zeros.  Rows stay 16-byte aligned.
bool head_size_ok(int64_t d) { return d >= 8 && d <= 128 && d % 8 == 0; }
int64_t padded_head_size(int64_t d) { return d <= 64 ? 64 : 128; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Launches `kernel` as a programmatic dependent of the work before it on the
// stream (cudaLaunchAttributeProgrammaticStreamSerialization): its blocks may
// start, and set up, while that work's last blocks run.  The kernels launched
// this way (forward, decode, elementwise chain) wait (griddepcontrol.wait)
// for the work before them to complete before they touch global memory.  The
// backward's three kernels are launched plainly: measured, their chain ran
// 1% slower as programmatic dependents.
template <typename... KParams, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KParams...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-device, per-kernel one-time set-up (opt-in shared memory size).
template <int D, bool CAUSAL, bool PAD, bool SNAKE>
cudaError_t prepare_kernel(int dev)
{
    static std::atomic<int> done[MAX_DEVICES];
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fa::fa_fwd_kernel<D, CAUSAL, PAD, SNAKE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)fa::Layout<D>::SMEM_BYTES);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

template <int D, bool CAUSAL, bool PAD, bool SNAKE>
fa_status launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const fa::Params& p, unsigned grid, int dev, cudaStream_t stream)
{
    if (prepare_kernel<D, CAUSAL, PAD, SNAKE>(dev) != cudaSuccess) return FA_ERR_CUDA;
    const cudaError_t e = launch_pdl(fa::fa_fwd_kernel<D, CAUSAL, PAD, SNAKE>, dim3(grid), dim3(fa::NUM_THREADS),
                                     fa::Layout<D>::SMEM_BYTES, stream, mq, mk, mv, p);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Causal problems run in cost order (snake) when `snake`; see item_of.
template <int D, bool CAUSAL, bool PAD = false>
fa_status launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                 const fa::Params& p, unsigned grid, int dev, cudaStream_t stream, bool snake)
{
    if constexpr (CAUSAL) {
        if (snake) return launch_one<D, true, PAD, true>(mq, mk, mv, p, grid, dev, stream);
    }
    return launch_one<D, CAUSAL, PAD, false>(mq, mk, mv, p, grid, dev, stream);
}

// Properties of a device that every call needs, queried once per device.
struct DevInfo {
    int sms;    // SMs: the persistent kernels run one CTA per SM
    int l2;     // L2 bytes: picks the causal item order
    bool sm103; // compute capability 10.3
};

std::atomic<int> g_devinfo_ready[MAX_DEVICES];
DevInfo g_devinfo[MAX_DEVICES];
std::mutex g_devinfo_lock;

// The current device (-1 if it cannot be queried) and its cached properties.
bool current_device(int* dev_out, DevInfo* info)
{
    int dev = -1;
    *dev_out = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return false;
    if (!g_devinfo_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> guard(g_devinfo_lock);
        if (!g_devinfo_ready[dev].load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0, l2 = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || sms <= 0)
                return false;
            g_devinfo[dev] = DevInfo{sms, l2, major == 10 && minor == 3};
            g_devinfo_ready[dev].store(1, std::memory_order_release);
        }
    }
    *dev_out = dev;
    *info = g_devinfo[dev];
    return true;
}

// FA_OK when the current device is an sm_103 (its properties in *info),
// FA_ERR_CUDA when it cannot be queried, FA_ERR_UNSUPPORTED otherwise.
fa_status sm103_device(int* dev, DevInfo* info)
{
    if (!current_device(dev, info)) return FA_ERR_CUDA;
    return info->sm103 ? FA_OK : FA_ERR_UNSUPPORTED;
}

// -------------------------------------------------------------- backward

template <int D, bool CAUSAL>
cudaError_t prepare_bwd_kernel(int dev)
{
    static std::atomic<int> done[MAX_DEVICES];
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fa::bwd::fa_bwd_kernel<D, CAUSAL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)fa::bwd::Layout<D>::SMEM_BYTES);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

struct BwdShape {
    int64_t BH, Np, num_kb, Dp;  // Dp: the kernel instance's (padded) head size
    size_t ws_bytes;
};

// Resident CTAs per SM of the elementwise kernel (cached per device).
template <bool WIDE>
int ew_ctas_per_sm(int dev)
{
    static std::atomic<int> cache[MAX_DEVICES];
    if (dev < 0 || dev >= MAX_DEVICES) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fa::ew::fa_bias_gelu_dropout_kernel<WIDE>,
                                                               fa::ew::THREADS, 0) == cudaSuccess)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

fa_status bwd_check(int64_t B, int64_t H, int64_t N, int64_t d, BwdShape* sh)
{
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (!head_size_ok(d)) return FA_ERR_UNSUPPORTED;
    const int64_t Dp = padded_head_size(d);
    const int64_t LIM = (int64_t)1 << 60;
    if (B > LIM / H || B * H > LIM / N || B * H * N > LIM / (Dp + 2)) return FA_ERR_INVALID_ARG;
    const int64_t BH = B * H;
    const int64_t Np = (N + fa::bwd::BQ - 1) / fa::bwd::BQ * fa::bwd::BQ;
    const int64_t num_kb = (N + fa::bwd::BKV - 1) / fa::bwd::BKV;
    // BH is the dQ conversion's grid.y; items are int
    if (Np > INT32_MAX / 2 || BH > 65535 || BH > (int64_t)(INT32_MAX / 2) / num_kb) return FA_ERR_INVALID_ARG;
    if (BH * Np > LIM / (Dp + 2)) return FA_ERR_INVALID_ARG;
    sh->BH = BH;
    sh->Np = Np;
    sh->num_kb = num_kb;
    sh->Dp = Dp;
    sh->ws_bytes = (size_t)(BH * Np) * (size_t)(Dp + 2) * sizeof(float);
    return FA_OK;
}

template <int D, bool CAUSAL>
fa_status launch_bwd_main(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                          const CUtensorMap& mdo, const CUtensorMap& mdq, const fa::bwd::Params& p, unsigned grid,
                          int dev, cudaStream_t st)
{
    if (prepare_bwd_kernel<D, CAUSAL>(dev) != cudaSuccess) return FA_ERR_CUDA;
    fa::bwd::fa_bwd_kernel<D, CAUSAL>
        <<<grid, fa::bwd::NUM_THREADS, fa::bwd::Layout<D>::SMEM_BYTES, st>>>(mq, mk, mv, mdo, mdq, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------- decode

// Query slots of the kernel instance serving nq query rows.
int decode_slots(int64_t nq) { return nq <= 1 ? 1 : nq <= 2 ? 2 : nq <= 4 ? 4 : 8; }

struct DecodePlan {
    int slots, splits, chunk;
    size_t ws_bytes;  // 0 when splits == 1 (the partial kernel writes the output)
};

// Splits of the key range.  Each CTA of the partial kernel streams one chunk
// (a whole number of rounds, at least 4) of one head's keys, and `wave` CTAs
// are resident at once.  All chunks cost about the same, so the cache is read
// in about (waves) x (chunk) time, waves = ceil(CTAs / wave): a last wave
// holding a few CTAs costs a whole chunk while most of the GPU idles.  Split
// results add traffic: the partial outputs are written and read back once.
// In bytes at the full bandwidth:
//   cost = waves * chunk * (K and V bytes a key) * wave + 2 * (partials' bytes).
// Candidates: 1 to 16 splits, and for k = 1 .. 8 the most splits that fill k
// waves.  The plan takes the candidate of least cost, or the smallest one
// within 2% of it.  A round is what the kernel instance for head size Dp
// (64 or 128) takes in one pass; the workspace holds d columns per partial
// output.
DecodePlan decode_plan(int64_t BH, int64_t nq, int64_t nk, int64_t d, int64_t wave)
{
    DecodePlan pl;
    pl.slots = decode_slots(nq);
    const int64_t Dp = padded_head_size(d);
    const int64_t round = fa::dec::WARPS * fa::dec::loads_in_flight(pl.slots) * (32 / (int)(Dp / 8));
    const int64_t max_splits = std::max<int64_t>(1, (nk + 4 * round - 1) / (4 * round));
    wave = std::max<int64_t>(1, wave);
    int64_t cand[24];
    int nc = 0;
    for (int64_t s = 1; s <= std::min<int64_t>(16, max_splits); ++s) cand[nc++] = s;
    for (int64_t k = 1; k <= 8; ++k) {
        const int64_t s = std::min<int64_t>(max_splits, k * wave / BH);
        if (s > cand[nc - 1]) cand[nc++] = s;  // ascending, no repeats
    }
    auto chunk_of = [&](int64_t s) { return ((nk + s - 1) / s + round - 1) / round * round; };
    double cost[24];
    double best = 0.0;
    for (int i = 0; i < nc; ++i) {
        const int64_t chunk = chunk_of(cand[i]), splits = (nk + chunk - 1) / chunk;
        const double partials = splits > 1 ? 2.0 * (double)(BH * nq * splits) * (double)(d + 1) * 4.0 : 0.0;
        cost[i] = (double)((BH * splits + wave - 1) / wave) * (double)chunk * (double)(4 * d) * (double)wave + partials;
        best = i == 0 ? cost[i] : std::min(best, cost[i]);
    }
    int pick = 0;
    while (cost[pick] > 1.02 * best) ++pick;
    const int64_t chunk = chunk_of(cand[pick]);
    const int64_t splits = (nk + chunk - 1) / chunk;
    pl.splits = (int)splits;
    pl.chunk = (int)chunk;
    pl.ws_bytes = splits > 1 ? (size_t)(BH * nq * splits) * (size_t)(d + 1) * sizeof(float) : 0;
    return pl;
}

// Checks of the sizes alone (no pointer, no device).
fa_status decode_check(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal)
{
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
    if (!head_size_ok(d)) return FA_ERR_UNSUPPORTED;
    if (Nq > fa::dec::MAX_NQ) return FA_ERR_UNSUPPORTED;
    const int64_t LIM = (int64_t)1 << 62;
    if (B > LIM / H || B * H > LIM / Nk || B * H * Nk > LIM / d) return FA_ERR_INVALID_ARG;
    if (B * H > 65535 || Nk > INT32_MAX / 2) return FA_ERR_INVALID_ARG;  // grid.y, key indices
    return FA_OK;
}

// Every check that needs no device: sizes, scale, null and misaligned
// pointers, outputs overlapping inputs.  The workspace is checked against
// the plan later (its size depends on the device).
fa_status decode_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int64_t B,
                      int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale, const void* ws)
{
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    const fa_status st = decode_check(B, H, Nq, Nk, d, causal);
    if (st != FA_OK) return st;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                          reinterpret_cast<uintptr_t>(ws);
    if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    const size_t qb = (size_t)(BH * Nq * d * 2), kb = (size_t)(BH * Nk * d * 2), lb = (size_t)(BH * Nq * 4);
    if (overlaps(o, qb, q, qb) || overlaps(o, qb, k, kb) || overlaps(o, qb, v, kb) || overlaps(o, qb, lse, lb) ||
        overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb))
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Resident CTAs per SM of the partial kernel instance serving `slots` query
// rows at head size d (cached per device); 0 if the query fails.
template <int D, int QM, bool PAD>
int dec_ctas_per_sm(int dev)
{
    static std::atomic<int> cache[MAX_DEVICES];
    if (dev < 0 || dev >= MAX_DEVICES) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fa::dec::fa_decode_partial_kernel<D, QM, PAD>,
                                                               fa::dec::THREADS, 0) == cudaSuccess)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <int D, bool PAD>
int dec_ctas_per_sm_d(int dev, int slots)
{
    switch (slots) {
    case 1: return dec_ctas_per_sm<D, 1, PAD>(dev);
    case 2: return dec_ctas_per_sm<D, 2, PAD>(dev);
    case 4: return dec_ctas_per_sm<D, 4, PAD>(dev);
    default: return dec_ctas_per_sm<D, 8, PAD>(dev);
    }
}

// The split plan on this device: one wave is the partial kernel's resident
// CTAs per SM times the SMs.  FA_ERR_CUDA if the occupancy query fails.
fa_status device_decode_plan(int dev, const DevInfo& info, int64_t BH, int64_t nq, int64_t nk, int64_t d,
                             DecodePlan* pl)
{
    const int slots = decode_slots(nq);
    const int per_sm = d == 128 ? dec_ctas_per_sm_d<128, false>(dev, slots)
                       : d == 64 ? dec_ctas_per_sm_d<64, false>(dev, slots)
                       : d > 64  ? dec_ctas_per_sm_d<128, true>(dev, slots)
                                 : dec_ctas_per_sm_d<64, true>(dev, slots);
    if (per_sm <= 0) return FA_ERR_CUDA;
    *pl = decode_plan(BH, nq, nk, d, (int64_t)per_sm * info.sms);
    return FA_OK;
}

template <int D, int QM, bool PAD>
fa_status launch_decode(const fa::dec::Params& p, int64_t BH, cudaStream_t st)
{
    if (launch_pdl(fa::dec::fa_decode_partial_kernel<D, QM, PAD>, dim3((unsigned)p.splits, (unsigned)BH),
                   dim3(fa::dec::THREADS), 0, st, p) != cudaSuccess)
        return FA_ERR_CUDA;
    if (p.splits > 1 &&
        launch_pdl(fa::dec::fa_decode_combine_kernel<D>, dim3((unsigned)(BH * p.nq)), dim3(D), 0, st, p) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

template <int D, bool PAD>
fa_status launch_decode_d(const fa::dec::Params& p, int slots, int64_t BH, cudaStream_t st)
{
    switch (slots) {
    case 1: return launch_decode<D, 1, PAD>(p, BH, st);
    case 2: return launch_decode<D, 2, PAD>(p, BH, st);
    case 4: return launch_decode<D, 4, PAD>(p, BH, st);
    default: return launch_decode<D, 8, PAD>(p, BH, st);
    }
}

// Decode with an explicit workspace (ws, ws_bytes >= the plan's), once the
// arguments have passed decode_args.
fa_status decode_run(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                     int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale, void* ws,
                     size_t ws_bytes, fa_stream_t stream)
{
    int dev = -1;
    DevInfo info;
    const fa_status ds = sm103_device(&dev, &info);
    if (ds != FA_OK) return ds;
    const int64_t BH = B * H;
    const size_t qb = (size_t)(BH * Nq * d * 2), kb = (size_t)(BH * Nk * d * 2), lb = (size_t)(BH * Nq * 4);
    DecodePlan pl;
    const fa_status ps = device_decode_plan(dev, info, BH, Nq, Nk, d, &pl);
    if (ps != FA_OK) return ps;
    if (pl.ws_bytes > 0) {
        if (!ws || ws_bytes < pl.ws_bytes) return FA_ERR_INVALID_ARG;
        if (overlaps(ws, pl.ws_bytes, o, qb) || overlaps(ws, pl.ws_bytes, lse, lb) || overlaps(ws, pl.ws_bytes, q, qb) ||
            overlaps(ws, pl.ws_bytes, k, kb) || overlaps(ws, pl.ws_bytes, v, kb))
            return FA_ERR_INVALID_ARG;
    }

    fa::dec::Params p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.ws_o = static_cast<float*>(ws);
    p.ws_lse = pl.ws_bytes > 0 ? static_cast<float*>(ws) + (size_t)(BH * Nq * pl.splits) * (size_t)d : nullptr;
    p.nq = (int)Nq;
    p.nk = (int)Nk;
    p.d = (int)d;
    p.splits = pl.splits;
    p.chunk = pl.chunk;
    p.causal = causal;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // Head sizes below 64 or 128 run in that instance with the columns past d
    // read as zeros (PAD).
    if (d == 128) return launch_decode_d<128, false>(p, pl.slots, BH, st);
    if (d == 64) return launch_decode_d<64, false>(p, pl.slots, BH, st);
    return d > 64 ? launch_decode_d<128, true>(p, pl.slots, BH, st) : launch_decode_d<64, true>(p, pl.slots, BH, st);
}

// Scratch of fa_decode_static: compiled into the library, one per device.
static __device__ __align__(256) unsigned char g_decode_scratch[FA_DECODE_STATIC_SCRATCH_BYTES];

// Device address of g_decode_scratch on device `dev` (the current device),
// looked up once per device.
void* static_scratch(int dev)
{
    static std::atomic<void*> cache[MAX_DEVICES];
    static std::mutex lock;
    if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
    void* p = cache[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> guard(lock);
    p = cache[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

// Clears the status bits a check has read (and the wait code, if it is still
// the one read), leaving bits that kernels on other streams set since.
__global__ void fa_clear_status_kernel(unsigned int bits, unsigned int where)
{
    atomicAnd(&fa::g_status, ~bits);
    atomicCAS(&fa::g_status_where, where, 0u);
}

}  // namespace

extern "C" {

fa_status fa_decode_static(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                           int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale,
                           fa_stream_t stream)
{
    // The argument checks come first, so that a call fa_decode would refuse
    // gets the same status here, whatever its sizes.
    const fa_status st = decode_args(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, nullptr);
    if (st != FA_OK) return st;
    int dev = -1;
    DevInfo info;
    const fa_status ds = sm103_device(&dev, &info);
    if (ds != FA_OK) return ds;
    DecodePlan pl;
    const fa_status ps = device_decode_plan(dev, info, B * H, Nq, Nk, d, &pl);
    if (ps != FA_OK) return ps;
    if (pl.ws_bytes > FA_DECODE_STATIC_SCRATCH_BYTES) return FA_ERR_TOO_LARGE;
    void* scratch = static_scratch(dev);
    if (!scratch) return FA_ERR_CUDA;
    return decode_run(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, scratch, FA_DECODE_STATIC_SCRATCH_BYTES,
                      stream);
}

fa_status fa_decode_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal,
                                    size_t* bytes)
{
    if (!bytes) return FA_ERR_INVALID_ARG;
    const fa_status st = decode_check(B, H, Nq, Nk, d, causal);
    if (st != FA_OK) return st;
    int dev = -1;
    DevInfo info;
    const fa_status ds = sm103_device(&dev, &info);
    if (ds != FA_OK) return ds;
    DecodePlan pl;
    const fa_status ps = device_decode_plan(dev, info, B * H, Nq, Nk, d, &pl);
    if (ps != FA_OK) return ps;
    *bytes = pl.ws_bytes;
    return FA_OK;
}

fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                    int64_t Nq, int64_t Nk, int64_t d, int causal, float scale, void* workspace,
                    size_t workspace_bytes, fa_stream_t stream)
{
    const fa_status st = decode_args(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, workspace);
    if (st != FA_OK) return st;
    return decode_run(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, workspace, workspace_bytes, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                 int64_t H, int64_t N, int64_t d, int causal, float scale, fa_stream_t stream)
{
    // ---- argument checks (no CUDA call before these pass)
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_INVALID_ARG;
    if (!head_size_ok(d)) return FA_ERR_UNSUPPORTED;
    const int64_t LIM = (int64_t)1 << 62;
    if (B > LIM / H || B * H > LIM / N || B * H * N > LIM / d) return FA_ERR_INVALID_ARG;
    const int64_t BH = B * H;
    const int64_t m_blocks = (N + fa::BM - 1) / fa::BM;
    if (BH > (((int64_t)1 << 31) - 1) / m_blocks) return FA_ERR_INVALID_ARG;
    if (N > INT32_MAX || BH > INT32_MAX) return FA_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_UNSUPPORTED;
    const size_t tb = (size_t)(BH * N * d * 2), lb = (size_t)(BH * N * 4);
    if (overlaps(o, tb, q, tb) || overlaps(o, tb, k, tb) || overlaps(o, tb, v, tb) ||
        overlaps(o, tb, lse, lb) || overlaps(lse, lb, q, tb) || overlaps(lse, lb, k, tb) ||
        overlaps(lse, lb, v, tb))
        return FA_ERR_INVALID_ARG;

    // ---- device
    int dev = -1;
    DevInfo info;
    const fa_status ds = sm103_device(&dev, &info);
    if (ds != FA_OK) return ds;

    CUtensorMap mq, mk, mv;
    if (!cached_map(&mq, q, BH, N, d, fa::BM) || !cached_map(&mk, k, BH, N, d, fa::BN) ||
        !cached_map(&mv, v, BH, N, d, fa::BN))
        return FA_ERR_CUDA;

    fa::Params p;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.N = (int)N;
    p.d = (int)d;
    p.num_m_blocks = (int)m_blocks;
    p.num_bh = (int)BH;
    p.num_items = (int)(BH * m_blocks);
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.debug_skip_k = g_debug_skip_k.load(std::memory_order_relaxed);
    // Causal items differ in cost.  Heavy/light pairs of a head keep its K/V
    // in L2 while its blocks run; when all heads' K and V fit in L2 anyway,
    // ordering the items by cost balances the CTAs better (see item_of).
    // (fa_debug_set_schedule may force either order for tests.)
    const double kv_bytes = 2.0 * (double)BH * (double)N * (double)d * 2.0;
    const int forced = g_debug_schedule.load(std::memory_order_relaxed);
    const bool snake = causal && (forced < 0 ? kv_bytes <= 0.6 * (double)info.l2 : forced == 1);
    // One CTA per SM, at most one per work item (per pair of items in pair order).
    const unsigned grid = (unsigned)std::min<int64_t>(snake ? BH * m_blocks : (BH * m_blocks + 1) / 2, info.sms);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    if (d == 128)
        return causal ? launch<128, true>(mq, mk, mv, p, grid, dev, st, snake)
                      : launch<128, false>(mq, mk, mv, p, grid, dev, st, snake);
    if (d == 64)
        return causal ? launch<64, true>(mq, mk, mv, p, grid, dev, st, snake)
                      : launch<64, false>(mq, mk, mv, p, grid, dev, st, snake);
    if (d > 64)
        return causal ? launch<128, true, true>(mq, mk, mv, p, grid, dev, st, snake)
                      : launch<128, false, true>(mq, mk, mv, p, grid, dev, st, snake);
    return causal ? launch<64, true, true>(mq, mk, mv, p, grid, dev, st, snake)
                  : launch<64, false, true>(mq, mk, mv, p, grid, dev, st, snake);
}

fa_status fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, size_t* bytes)
{
    if (!bytes) return FA_ERR_INVALID_ARG;
    BwdShape sh;
    const fa_status st = bwd_check(B, H, N, d, &sh);
    if (st != FA_OK) return st;
    *bytes = sh.ws_bytes;
    return FA_OK;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream)
{
    // ---- argument checks (no CUDA call before these pass)
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_INVALID_ARG;
    BwdShape sh;
    const fa_status chk = bwd_check(B, H, N, d, &sh);
    if (chk != FA_OK) return chk;
    if (workspace_bytes < sh.ws_bytes) return FA_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                          reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                          reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv) |
                          reinterpret_cast<uintptr_t>(workspace);
    if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_UNSUPPORTED;
    const int64_t BH = sh.BH;
    const size_t tb = (size_t)(BH * N * d * 2), lb = (size_t)(BH * N * 4);
    // Outputs and the workspace may overlap no input and no other output.
    const void* ins[6] = {q, k, v, o, lse, dout};
    const size_t in_b[6] = {tb, tb, tb, tb, lb, tb};
    const void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_b[4] = {tb, tb, tb, sh.ws_bytes};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_b[a], ins[b], in_b[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_b[a], outs[b], out_b[b])) return FA_ERR_INVALID_ARG;
    }

    // ---- device
    int dev = -1;
    DevInfo info;
    const fa_status ds = sm103_device(&dev, &info);
    if (ds != FA_OK) return ds;
    const int sms = info.sms;
    float* const lse2 = static_cast<float*>(workspace);
    float* const dsum = lse2 + BH * sh.Np;
    float* const acc = dsum + BH * sh.Np;
    CUtensorMap mq, mk, mv, mdo, mdq;
    if (!cached_map(&mq, q, BH, N, d, fa::bwd::BQ) || !cached_map(&mk, k, BH, N, d, fa::bwd::BKV) ||
        !cached_map(&mv, v, BH, N, d, fa::bwd::BKV) || !cached_map(&mdo, dout, BH, N, d, fa::bwd::BQ) ||
        !make_acc_map(&mdq, acc, BH, sh.Np, sh.Dp))
        return FA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // 1. D, L * log2 e, zeroed dQ accumulator.
    const int64_t rows = BH * sh.Np;
    fa::bwd::fa_bwd_prep_kernel<<<(unsigned)((rows + 8 * fa::bwd::PREP_ROWS - 1) / (8 * fa::bwd::PREP_ROWS)), 256, 0,
                                   st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, lse2, dsum, acc,
        (int)N, (int)sh.Np, (int)d, (int)sh.Dp, rows);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

    // 2. dK, dV and the dQ accumulator.
    fa::bwd::Params p;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.lse2 = lse2;
    p.dsum = dsum;
    p.dq_acc = acc;
    p.N = (int)N;
    p.d = (int)d;
    p.Np = (int)sh.Np;
    p.num_kb = (int)sh.num_kb;
    p.num_items = (int)(BH * sh.num_kb);
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.scale = scale;
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.debug_skip_q = g_debug_skip_k.load(std::memory_order_relaxed);
    const unsigned grid = (unsigned)std::min<int64_t>((BH * sh.num_kb + 1) / 2, sms);
    fa_status ms;
    if (sh.Dp == 128)
        ms = causal ? launch_bwd_main<128, true>(mq, mk, mv, mdo, mdq, p, grid, dev, st)
                    : launch_bwd_main<128, false>(mq, mk, mv, mdo, mdq, p, grid, dev, st);
    else
        ms = causal ? launch_bwd_main<64, true>(mq, mk, mv, mdo, mdq, p, grid, dev, st)
                    : launch_bwd_main<64, false>(mq, mk, mv, mdo, mdq, p, grid, dev, st);
    if (ms != FA_OK) return ms;

    // 3. dQ = scale * accumulator, bf16.
    const int64_t n8 = BH * N * d / 8;
    fa::bwd::fa_bwd_dq_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(
        acc, static_cast<__nv_bfloat16*>(dq), (int)N, (int)sh.Np, (int)d, (int)sh.Dp, n8, scale);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bias_gelu_dropout(const void* x, const void* bias, const uint32_t* keep, void* y, int64_t rows,
                               int64_t cols, float p, fa_stream_t stream)
{
    // ---- argument checks (no CUDA call before these pass)
    if (!x || !bias || !y) return FA_ERR_INVALID_ARG;
    if (rows < 1 || cols < 1 || !(p >= 0.0f && p < 1.0f)) return FA_ERR_INVALID_ARG;
    if (cols % 8 != 0) return FA_ERR_UNSUPPORTED;
    if (rows > ((int64_t)1 << 62) / cols || cols / 8 > INT32_MAX) return FA_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(bias) |
                          reinterpret_cast<uintptr_t>(y);
    if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(keep) & 3u) != 0) return FA_ERR_UNSUPPORTED;
    const int64_t n = rows * cols;
    const size_t tb = (size_t)n * 2, bb = (size_t)cols * 2, kb = (size_t)((n + 31) / 32) * 4;
    if (overlaps(y, tb, x, tb) || overlaps(y, tb, bias, bb) || (keep && overlaps(y, tb, keep, kb)))
        return FA_ERR_INVALID_ARG;

    int dev = -1;
    DevInfo info;
    const fa_status ds = sm103_device(&dev, &info);
    if (ds != FA_OK) return ds;
    const int sms = info.sms;

    fa::ew::Params prm;
    prm.x = static_cast<const __nv_bfloat16*>(x);
    prm.bias = static_cast<const __nv_bfloat16*>(bias);
    prm.keep = reinterpret_cast<const uint8_t*>(keep);
    prm.y = static_cast<__nv_bfloat16*>(y);
    prm.n8 = n / 8;
    prm.cols8 = (int)(cols / 8);
    // Division by the invariant cols8 (Granlund and Montgomery's round-up
    // method for 31-bit numerators): magic = floor(2^(31+l) / cols8) + 1.
    int l = 0;
    while (((int64_t)1 << l) < (int64_t)prm.cols8) ++l;
    prm.magic = (uint32_t)((((uint64_t)1) << (31 + l)) / (uint64_t)prm.cols8 + 1);
    prm.shift = 31 + l;
    prm.scale = 1.0f / (1.0f - p);
    // Exactly the CTAs that are resident at once (one wave), each thread
    // keeping UNROLL 16-byte loads in flight, walking the tensor grid-stride.
    const bool wide = prm.n8 >= ((int64_t)1 << 31);
    const int per_sm = wide ? ew_ctas_per_sm<true>(dev) : ew_ctas_per_sm<false>(dev);
    if (per_sm <= 0) return FA_ERR_CUDA;
    const int64_t per_cta = (int64_t)fa::ew::THREADS * fa::ew::UNROLL;
    const unsigned grid =
        (unsigned)std::max<int64_t>(1, std::min<int64_t>((prm.n8 + per_cta - 1) / per_cta, (int64_t)per_sm * sms));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        wide ? launch_pdl(fa::ew::fa_bias_gelu_dropout_kernel<true>, dim3(grid), dim3(fa::ew::THREADS), 0, st, prm)
             : launch_pdl(fa::ew::fa_bias_gelu_dropout_kernel<false>, dim3(grid), dim3(fa::ew::THREADS), 0, st, prm);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_check_device_status(fa_stream_t stream, uint32_t* where)
{
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned int h[2] = {0u, 0u};
    if (cudaMemcpyFromSymbolAsync(&h[0], fa::g_status, sizeof(unsigned int), 0,
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&h[1], fa::g_status_where, sizeof(unsigned int), 0,
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return FA_ERR_CUDA;
    if (where) *where = h[1];
    if (h[0] != 0u) {
        const fa_status st_code = (h[0] & fa::STATUS_TIMEOUT) ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
        // Clear what was read, atomically on the device: a bit that a kernel
        // on another stream set in between stays for the next check.
        fa_clear_status_kernel<<<1, 1, 0, st>>>(h[0], h[1]);
        if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
        return st_code;
    }
    return FA_OK;
}

fa_status fa_get_device_status(fa_stream_t stream) { return fa_check_device_status(stream, nullptr); }

fa_status fa_set_wait_limit_ns(uint64_t ns)
{
    g_wait_limit_ns.store(ns ? ns : DEFAULT_WAIT_LIMIT_NS, std::memory_order_relaxed);
    return FA_OK;
}

fa_status fa_debug_skip_k_tile(int tile)
{
    if (tile < -1) return FA_ERR_INVALID_ARG;
    g_debug_skip_k.store(tile, std::memory_order_relaxed);
    return FA_OK;
}

fa_status fa_debug_decode_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t wave, int* splits,
                               int* chunk)
{
    if (!splits || !chunk || wave < 1) return FA_ERR_INVALID_ARG;
    const fa_status st = decode_check(B, H, Nq, Nk, d, 0);
    if (st != FA_OK) return st;
    const DecodePlan pl = decode_plan(B * H, Nq, Nk, d, wave);
    *splits = pl.splits;
    *chunk = pl.chunk;
    return FA_OK;
}

fa_status fa_debug_set_schedule(int order)
{
    if (order < -1 || order > 1) return FA_ERR_INVALID_ARG;
    g_debug_schedule.store(order, std::memory_order_relaxed);
    return FA_OK;
}

const char* fa_status_string(fa_status s)
{
    switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported (head size, alignment or device)";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case FA_ERR_TOO_LARGE: return "the sizes need more scratch than the library's static array holds";
    }
    return "unknown status";
}

int fa_version(void) { return FA_VERSION; }

#ifdef FA_TRACE
// Trace builds only: points the kernels' event trace at a device buffer.
int fa_debug_set_trace(void* device_buffer)
{
    unsigned long long* p = static_cast<unsigned long long*>(device_buffer);
    return cudaMemcpyToSymbol(fa::g_trace, &p, sizeof p) == cudaSuccess ? 0 : 1;
}
#endif

}  // extern "C"
