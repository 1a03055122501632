// Attention for decode on sm_103a: a few query rows against a long KV cache.
//
// "Fusion and IO-aware kernels" (section "Where it breaks"): with one query
// token per sequence, attention is dominated by reading the KV cache, not by
// the score matrix, and split-K variants (FlashDecoding) parallelise across
// the sequence instead.  So the cache is cut into `splits` chunks; one CTA
// per (head, chunk) streams its chunk of K and V once from HBM and carries
// the online-softmax state ("Kernels — fusion and FlashAttention" §3) over
// it, then writes its normalised partial output o_s and logsumexp lse_s.  A
// second kernel merges the chunks of each query row exactly:
//
//   lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) * o_s.
//
// Query i stands at key position Nk - Nq + i: under the causal mask it sees
// keys 0 .. Nk - Nq + i.
//
// The work is a bandwidth problem: 4 * Nq * d FLOPs per 4 * d bytes of K and
// V, i.e. about Nq FLOP per byte.  Up to 8 query rows, a 128-row tensor-core
// tile would be almost all padding, so the dot products run on the CUDA
// cores in fp32 (bf16 inputs widened exactly; the probabilities are not
// rounded).  Loads: a group of G = d/8 lanes owns one key row (16 bytes per
// lane, one coalesced row per group), and every lane keeps U rows of K and of
// V in flight.
//
// Head sizes d below D (multiples of 8) run in the D = 64 or 128 instance
// with PAD: rows are d elements apart, the lanes whose 8 columns lie past d
// load nothing and hold zeros (which add nothing to any dot product), and
// only d columns are written.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fa {
namespace dec {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int MAX_NQ = 8;
constexpr float LN2 = 0.69314718055994530942f;

// Loads in flight per lane shrink as the query rows (registers per key) grow.
constexpr int loads_in_flight(int qm) { return qm <= 2 ? 8 : (qm <= 4 ? 4 : 2); }

template <int D, int QM>
struct Cfg {
    static_assert(D == 64 || D == 128, "head size");
    static_assert(QM >= 1 && QM <= MAX_NQ, "query rows");
    static constexpr int G = D / 8;                     // lanes per key row
    static constexpr int KPW = 32 / G;                  // key rows per warp load
    static constexpr int U = loads_in_flight(QM);       // rows of K (and of V) in flight per lane
    static constexpr int ROUND = WARPS * U * KPW;       // keys per CTA round
};

struct Params {
    const __nv_bfloat16* q;  // (B*H, Nq, d)
    const __nv_bfloat16* k;  // (B*H, Nk, d)
    const __nv_bfloat16* v;
    __nv_bfloat16* o;        // (B*H, Nq, d), written when splits == 1
    float* lse;              // (B*H, Nq), written when splits == 1
    float* ws_o;             // (B*H*Nq, splits, d) partial outputs (normalised)
    float* ws_lse;           // (B*H*Nq, splits) partial logsumexps (natural log)
    int nq, nk, splits, chunk;  // chunk: keys per split (a multiple of ROUND)
    int d;                   // the caller's head size (<= D): row stride and columns present
    int causal;
    float scale_log2;        // scale * log2(e)
};

__device__ __forceinline__ void unpack8(const uint4 w, float (&f)[8])
{
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xFFFF0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint4 ldg_stream(const __nv_bfloat16* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Partial attention of one (head, chunk) for QM query slots (Nq <= QM).
template <int D, int QM, bool PAD>
__global__ void __launch_bounds__(THREADS)
    fa_decode_partial_kernel(const Params p)
{
    ptx::griddep_wait();  // a programmatic dependent: the inputs are complete
    ptx::griddep_launch_dependents();
    using C = Cfg<D, QM>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / C::G, sub = lane % C::G;  // key of the load, 8 columns of it
    const int split = blockIdx.x, bh = blockIdx.y;
    const int nq = p.nq, nk = p.nk;
    const int k_begin = split * p.chunk;
    const int k_end = min(nk, k_begin + p.chunk);
    const int dd = PAD ? p.d : D;              // row stride and columns present
    const bool cols_ok = !PAD || sub * 8 < dd;  // this lane's columns exist

    // This lane's 8 columns of each query row, times scale * log2(e).
    float qv[QM][8];
#pragma unroll
    for (int i = 0; i < QM; ++i) {
        if (i < nq && cols_ok) {
            const uint4 w = *reinterpret_cast<const uint4*>(p.q + ((int64_t)bh * nq + i) * dd + sub * 8);
            unpack8(w, qv[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[i][e] *= p.scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[i][e] = 0.f;
        }
    }
    // Online-softmax state of this lane group's keys (base 2), per query.
    float m[QM], l[QM], acc[QM][8];
#pragma unroll
    for (int i = 0; i < QM; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
    }

    const __nv_bfloat16* const kh = p.k + (int64_t)bh * nk * dd + sub * 8;
    const __nv_bfloat16* const vh = p.v + (int64_t)bh * nk * dd + sub * 8;
    for (int r0 = k_begin; r0 < k_end; r0 += C::ROUND) {
        // Key of load u: rows of one warp are consecutive (KPW per load).
        uint4 kw[C::U], vw[C::U];
        int key[C::U];
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
            key[u] = r0 + (warp * C::U + u) * C::KPW + grp;
            const int kc = min(key[u], k_end - 1);  // rows past the chunk: a valid row, masked below
            kw[u] = cols_ok ? ldg_stream(kh + (int64_t)kc * dd) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
            const int kc = min(key[u], k_end - 1);
            vw[u] = cols_ok ? ldg_stream(vh + (int64_t)kc * dd) : make_uint4(0u, 0u, 0u, 0u);
        }
        // Scores s[i][u] (base 2), reduced over the G lanes of the group.
        float s[QM][C::U];
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
            float kf[8];
            unpack8(kw[u], kf);
#pragma unroll
            for (int i = 0; i < QM; ++i) {
                float t = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) t = fmaf(qv[i][e], kf[e], t);
#pragma unroll
                for (int off = C::G / 2; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
                const bool visible = key[u] < k_end && (!p.causal || key[u] <= nk - nq + i);
                s[i][u] = visible ? t : -INFINITY;
            }
        }
#pragma unroll
        for (int i = 0; i < QM; ++i) {
            float mx = s[i][0];
#pragma unroll
            for (int u = 1; u < C::U; ++u) mx = fmaxf(mx, s[i][u]);
            if (mx > m[i]) {  // the running max rises: rescale what was summed
                const float corr = ex2f(m[i] - mx);  // 0 on the first visible key
                l[i] *= corr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] *= corr;
                m[i] = mx;
            }
        }
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
            float vf[8];
            unpack8(vw[u], vf);
#pragma unroll
            for (int i = 0; i < QM; ++i) {
                const float pr = (s[i][u] == -INFINITY) ? 0.f : ex2f(s[i][u] - m[i]);
                l[i] += pr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pr, vf[e], acc[i][e]);
            }
        }
    }

    // Merge the KPW lane groups of the warp (lanes sub, sub + G, ... hold the
    // same columns).
#pragma unroll
    for (int off = C::G; off < 32; off <<= 1) {
#pragma unroll
        for (int i = 0; i < QM; ++i) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[i], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[i], off);
            const float mn = fmaxf(m[i], mo);
            const float ca = (m[i] == -INFINITY) ? 0.f : ex2f(m[i] - mn);
            const float cb = (mo == -INFINITY) ? 0.f : ex2f(mo - mn);
            l[i] = l[i] * ca + lo * cb;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[i][e], off);
                acc[i][e] = acc[i][e] * ca + ao * cb;
            }
            m[i] = mn;
        }
    }

    // Merge the warps through shared memory.
    __shared__ float sm_m[WARPS][QM], sm_l[WARPS][QM];
    __shared__ float sm_o[WARPS][QM][D];
    if (lane < C::G) {
#pragma unroll
        for (int i = 0; i < QM; ++i) {
            if (lane == 0) {
                sm_m[warp][i] = m[i];
                sm_l[warp][i] = l[i];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) sm_o[warp][i][sub * 8 + e] = acc[i][e];
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < QM * D; t += THREADS) {
        const int i = t / D, c = t % D;
        if (i >= nq || c >= dd) continue;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mx = fmaxf(mx, sm_m[w][i]);
        float lt = 0.f, ot = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const float cw = (sm_m[w][i] == -INFINITY) ? 0.f : ex2f(sm_m[w][i] - mx);
            lt += sm_l[w][i] * cw;
            ot += sm_o[w][i][c] * cw;
        }
        const int64_t row = (int64_t)bh * nq + i;
        // lse in natural log; a chunk whose keys this query does not see
        // (causal) has lt = 0: lse_s = -inf, weight 0 in the merge.
        const float lse_s = (lt > 0.f) ? (mx + __log2f(lt)) * LN2 : -INFINITY;
        const float o_s = (lt > 0.f) ? ot / lt : 0.f;
        if (p.splits == 1) {
            p.o[row * dd + c] = __float2bfloat16_rn(o_s);
            if (c == 0) p.lse[row] = lse_s;
        } else {
            p.ws_o[(row * p.splits + split) * dd + c] = o_s;
            if (c == 0) p.ws_lse[row * p.splits + split] = lse_s;
        }
    }
}

// Merge of the splits of one query row: block of D threads, one column each
// (the columns past the head size d idle).
template <int D>
__global__ void __launch_bounds__(D) fa_decode_combine_kernel(const Params p)
{
    ptx::griddep_wait();  // a programmatic dependent: the partial results are complete
    ptx::griddep_launch_dependents();
    const int64_t row = blockIdx.x;  // (bh, query)
    const int c = threadIdx.x;
    const int dd = p.d;
    if (c >= dd) return;
    const float* const ls = p.ws_lse + row * p.splits;
    float mx = -INFINITY;
    for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, ls[s]);
    float wsum = 0.f, ot = 0.f;
    for (int s = 0; s < p.splits; ++s) {
        const float w = (ls[s] == -INFINITY) ? 0.f : __expf(ls[s] - mx);
        wsum += w;
        ot += w * p.ws_o[(row * p.splits + s) * dd + c];
    }
    p.o[row * dd + c] = __float2bfloat16_rn(ot / wsum);
    if (c == 0) p.lse[row] = mx + __logf(wsum);
}

}  // namespace dec
}  // namespace fa
