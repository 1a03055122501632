// Fused elementwise chain for sm_103a: y = dropout(gelu(x + bias)), bf16.
//
// "Fusion and IO-aware kernels", § The idea in one minute: a bias add, a GELU
// and a dropout run as three kernels move the tensor six times; fused, the
// tensor is read once and written once, and the arithmetic in between stays
// in registers.  For element (r, c), flat index e = r*cols + c:
//
//   h = x[r][c] + bias[c]
//   g = 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3)))   ("Writing and
//       Benchmarking Custom Kernels" §10.2.1, the tanh form of GELU)
//   y = keep(e) ? g / (1 - p) : 0
//
// keep(e) is bit e % 32 of word e / 32 of a packed mask that the caller
// draws (the dropout's random numbers are an input).
//
// The work is HBM-bound (4.125 bytes per element against ~15 flops), so the
// kernel is built around the memory system: each thread moves 16-byte vectors
// of 8 elements, keeps UNROLL of them in flight, and a grid sized to the SM
// count walks the tensor in a grid-stride loop.  A vector never crosses a
// row (cols is a multiple of 8), its bias is one 16-byte load (L1/L2
// resident), and its 8 keep bits are one byte of the mask.
//
// GELU is evaluated through the identity 0.5 h (1 + tanh a) = h / (1 + e^(-2a)):
// one ex2 and one reciprocal on the special-function unit, with the exponent
// clamped at 64 (the value is then below 2^-64 |h|) so the reciprocal never
// sees an infinity.  Unlike tanh.approx, this keeps its relative accuracy on
// the negative side, where 1 + tanh a cancels.  The rest is packed fp32x2
// arithmetic on element pairs, and the dropout is branch-free: the keep bit
// selects the element's factor, 1/(1 - p) or 0.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fa {
namespace ew {

constexpr int THREADS = 256;
constexpr int UNROLL = 4;  // 16-byte vectors in flight per thread

struct Params {
    const __nv_bfloat16* x;
    const __nv_bfloat16* bias;
    const uint8_t* keep;  // packed keep bits viewed as bytes (byte v: elements 8v .. 8v+7); null: keep all
    __nv_bfloat16* y;
    int64_t n8;           // vectors of 8 elements (rows * cols / 8)
    int cols8;            // cols / 8
    uint32_t magic;       // v / cols8 = (v * magic) >> shift for v < 2^31 (division by an invariant integer)
    int shift;
    float scale;          // 1 / (1 - p)
};

// Column vector of vector v.  Below 2^31 vectors, the quotient v / cols8 comes
// from one 64-bit multiply with the host's magic number (Granlund and
// Montgomery's round-up method: magic = floor(2^(31+l) / cols8) + 1,
// l = ceil(log2 cols8), exact for every v < 2^31); WIDE falls back to a
// 64-bit remainder.
template <bool WIDE>
__device__ __forceinline__ int col8_of(int64_t v, const Params& p)
{
    if (WIDE) return (int)(v % p.cols8);
    const uint32_t q = (uint32_t)(((uint64_t)v * p.magic) >> p.shift);
    return (int)((uint32_t)v - q * (uint32_t)p.cols8);
}

// -2 log2(e) sqrt(2/pi) and 0.044715 times it: 2^(h (K1 + K2 h^2)) = e^(-2a).
constexpr float K1 = -2.0f * 1.4426950408889634f * 0.7978845608028654f;
constexpr float K2 = K1 * 0.044715f;

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two neighbouring elements (a bf16 pair of x and of the bias, their two keep
// bits as the pair's dropout factors {0 or 1/(1-p)} x 2) -> a bf16 pair of y.
__device__ __forceinline__ uint32_t chain2(uint32_t xw, uint32_t bw, uint64_t fac)
{
    const uint64_t x2 = ptx::f2_pack(__uint_as_float(xw << 16), __uint_as_float(xw & 0xFFFF0000u));
    const uint64_t b2 = ptx::f2_pack(__uint_as_float(bw << 16), __uint_as_float(bw & 0xFFFF0000u));
    const uint64_t h = ptx::f2_add(x2, b2);
    const uint64_t w = ptx::f2_fma(ptx::f2_pack(K2, K2), ptx::f2_mul(h, h), ptx::f2_pack(K1, K1));
    float z0, z1;
    ptx::f2_unpack(ptx::f2_mul(h, w), z0, z1);
    const uint64_t den = ptx::f2_add(ptx::f2_pack(ptx::ex2(fminf(z0, 64.0f)), ptx::ex2(fminf(z1, 64.0f))),
                                     ptx::f2_pack(1.0f, 1.0f));
    float d0, d1;
    ptx::f2_unpack(den, d0, d1);
    const uint64_t y = ptx::f2_mul(ptx::f2_mul(h, fac), ptx::f2_pack(rcp_approx(d0), rcp_approx(d1)));
    float y0, y1;
    ptx::f2_unpack(y, y0, y1);
    return ptx::pack_bf16x2(y0, y1);
}

template <bool WIDE>
__global__ void __launch_bounds__(THREADS, 4) fa_bias_gelu_dropout_kernel(const Params p)
{
    ptx::griddep_wait();  // a programmatic dependent: the inputs are complete
    ptx::griddep_launch_dependents();
    // Dropout factors of an element pair, indexed by its two keep bits.
    __shared__ uint64_t ftab[4];
    if (threadIdx.x < 4)
        ftab[threadIdx.x] = ptx::f2_pack((threadIdx.x & 1u) ? p.scale : 0.0f, (threadIdx.x & 2u) ? p.scale : 0.0f);
    __syncthreads();
    const int64_t per_round = (int64_t)gridDim.x * THREADS * UNROLL;
    for (int64_t v0 = (int64_t)blockIdx.x * THREADS * UNROLL + threadIdx.x; v0 < p.n8; v0 += per_round) {
        uint4 xv[UNROLL];
        uint32_t kb[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t v = v0 + (int64_t)u * THREADS;
            if (v < p.n8) {
                xv[u] = ld_stream(p.x + v * 8);
                kb[u] = p.keep ? (uint32_t)__ldg(p.keep + v) : 0xFFu;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t v = v0 + (int64_t)u * THREADS;
            if (v < p.n8) {
                // The bias (L1/L2-resident) is loaded here, so that its registers
                // hold no vector in flight.
                const uint4 bv = __ldg(reinterpret_cast<const uint4*>(p.bias) + col8_of<WIDE>(v, p));
                const uint32_t w0 = chain2(xv[u].x, bv.x, ftab[kb[u] & 3u]);
                const uint32_t w1 = chain2(xv[u].y, bv.y, ftab[(kb[u] >> 2) & 3u]);
                const uint32_t w2 = chain2(xv[u].z, bv.z, ftab[(kb[u] >> 4) & 3u]);
                const uint32_t w3 = chain2(xv[u].w, bv.w, ftab[(kb[u] >> 6) & 3u]);
                // Streaming store: y is not read again by this kernel.
                asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p.y + v * 8), "r"(w0), "r"(w1),
                             "r"(w2), "r"(w3)
                             : "memory");
            }
        }
    }
}

}  // namespace ew
}  // namespace fa
