/*
 * fa.h — C ABI of the GB300 (sm_103a) attention-forward library.
 *
 * The library computes, for every (batch b, head h) and query row i,
 *
 *     O_i = sum_j softmax_j(scale * q_i . k_j  [ -inf where causal and j > i ]) * v_j
 *     L_i = ln sum_j exp(scale * q_i . k_j)   (over the keys row i may see)
 *
 * without ever writing the N x N score matrix to device memory: query rows
 * are taken 128 at a time, K/V tiles stream through shared memory, and an
 * online-softmax state (running max m, running denominator l, output
 * accumulator o, rescaled by exp(m_old - m_new) when the max rises) is
 * carried per row, as "Kernels — fusion and FlashAttention" §3–§4 and
 * "Fusion and IO-aware kernels" § FlashAttention (steps 1–4) describe.  The
 * saved logsumexp is the m + log l statistic of "Kernels — fusion and
 * FlashAttention" §5 and "Writing and Benchmarking Custom Kernels" §10.3.2,
 * kept in fp32.
 *
 * Every function returns an fa_status; none throws, aborts or prints.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same type as cudaStream_t / CUstream); NULL is
 * the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *fa_stream_t;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, non-finite or non-positive
                                scale, causal not 0/1, o overlapping q/k/v/lse */
    FA_ERR_UNSUPPORTED = 2,  /* head size not supported, pointer not 16-byte aligned
                                (lse: 4-byte), device not sm_103 */
    FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or the launch failed */
    FA_ERR_TIMEOUT = 4,      /* a kernel gave up a pipeline wait (device status) */
    FA_ERR_TOO_LARGE = 5     /* fa_decode_static: the sizes need more scratch than
                                FA_DECODE_STATIC_SCRATCH_BYTES */
} fa_status;

/*
 * fa_fwd — attention forward on one GPU.
 *
 * Operation: see the file comment ("Kernels — fusion and FlashAttention" §2
 * for the attention itself, §3 for the recurrence; "Writing and Benchmarking
 * Custom Kernels" §10.3.1 for causal tile skipping and the masked last tile).
 *
 * Arguments
 *   q, k, v  device pointers, bf16, contiguous (B, H, N, d) row-major, read only.
 *   o        device pointer, bf16, contiguous (B, H, N, d); fully written.
 *   lse      device pointer, fp32, contiguous (B, H, N); fully written with the
 *            natural-log logsumexp of the scaled, masked scores of each row.
 *   B, H, N  batch, heads, sequence length (queries = keys = N); each >= 1,
 *            B*H*N*d < 2^62, B*H*ceil(N/128) < 2^31.
 *   d        head size: a multiple of 8 from 8 to 128.  64 and 128 run
 *            natively; other sizes run in the 64- or 128-column kernel with
 *            the columns past d read as zeros by the TMA loads (they add
 *            nothing to any dot product), and only d columns of O are written.
 *   causal   0: every query sees every key; 1: query i sees keys 0..i.
 *   scale    finite, > 0 (typically 1/sqrt(d)); scores are scale * q.k.
 *   stream   CUDA stream the work is enqueued on.
 *
 * Ownership: the caller allocates and frees every buffer.  The library keeps
 * no per-call state and allocates no device memory.  It caches one-time
 * per-device set-up (kernel attributes, the SM count and L2 size) and, per
 * host thread, the TMA descriptors of the last few buffers it was given (a
 * descriptor is a pure function of the address and sizes, so a reused
 * buffer gets the same descriptor a fresh encode would give).
 *
 * Asynchrony: returns after enqueuing; results are valid once `stream` has
 * been synchronised.  Errors found before the launch are returned directly;
 * a pipeline timeout inside the kernel is reported by fa_check_device_status.
 * o and lse must not overlap q, k, v or each other (FA_ERR_INVALID_ARG).
 * The kernel is launched as a programmatic dependent of the work before it
 * on `stream` (CUDA programmatic dependent launch): its blocks may start and
 * set up while that work's last blocks run, but read and write device memory
 * only once it has completed, so stream order holds as for a plain launch.
 * The device is the calling thread's current device.
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                 int64_t H, int64_t N, int64_t d, int causal, float scale, fa_stream_t stream);

/*
 * fa_decode_workspace_bytes — workspace that fa_decode needs for these sizes
 * on the current device (0 when the key range is not split).  Arguments as
 * for fa_decode.  FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED as fa_decode
 * reports them; FA_ERR_CUDA if the device cannot be queried.
 */
fa_status fa_decode_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                                    int causal, size_t *bytes);

/*
 * fa_decode — attention of a few query rows against a long key/value cache
 * ("Fusion and IO-aware kernels", section "Where it breaks": decode reads the
 * whole KV cache per query token; split-K variants (FlashDecoding)
 * parallelise across the sequence).  The key range is cut into chunks, each
 * chunk's online softmax ("Kernels — fusion and FlashAttention" §3) gives a
 * partial output and logsumexp, and the chunks are merged exactly by their
 * logsumexps.
 *
 * For query row i of (b, h):
 *     O_i = sum_j softmax_j(scale * q_i . k_j) * v_j,  L_i = ln sum_j exp(scale * q_i . k_j)
 * over keys j = 0 .. Nk-1, or, with causal = 1, j = 0 .. Nk - Nq + i (query i
 * stands at position Nk - Nq + i: the newest Nq keys belong to the queries).
 *
 * Arguments
 *   q        device pointer, bf16, contiguous (B, H, Nq, d); 1 <= Nq <= 8.
 *   k, v     device pointers, bf16, contiguous (B, H, Nk, d): the cache.
 *   o        device pointer, bf16, contiguous (B, H, Nq, d); fully written.
 *   lse      device pointer, fp32, contiguous (B, H, Nq); fully written.
 *   B, H     batch and heads, B*H <= 65535.  causal: 0 or 1 (1 requires
 *            Nq <= Nk).  scale: finite, > 0.
 *   d        head size: a multiple of 8 from 8 to 128, as for fa_fwd (sizes
 *            other than 64 and 128 run in the 64- or 128-column kernel with
 *            the columns past d read as zeros; only d columns are written).
 *   workspace, workspace_bytes
 *            device scratch of at least fa_decode_workspace_bytes(...) bytes,
 *            16-byte aligned (may be NULL when that size is 0).  It holds the
 *            chunks' partial results between the two kernels of one call and
 *            must not be shared by calls that may run at the same time.
 *   stream   CUDA stream the work is enqueued on.
 *
 * Ownership: the caller allocates every buffer, including the workspace; the
 * library allocates nothing.  Asynchrony and launches as for fa_fwd (both
 * kernels).  Errors: as fa_fwd,
 * plus FA_ERR_INVALID_ARG for a missing or short workspace, and
 * FA_ERR_UNSUPPORTED for Nq > 8 or a workspace that is not 16-byte aligned.
 * The sizes, scale, pointers and overlaps with the inputs are checked before
 * the device is queried.
 */
fa_status fa_decode(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                    int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale,
                    void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_decode_static — fa_decode without a caller workspace and without any
 * allocation.  The pages have no counterpart to this entry point: it exists
 * for callers that cannot hand over device memory at the point of the call,
 * for instance a runtime whose own pool already owns all device memory, or
 * code that must not call cudaMalloc/cudaFree because those calls can
 * synchronise the device.  The chunks' partial results go to a scratch array
 * compiled into the library (a static device array of
 * FA_DECODE_STATIC_SCRATCH_BYTES, 8 MiB), so nothing is allocated by this
 * call or by the library.
 *
 *   - Arguments, results and errors are those of fa_decode, minus the
 *     workspace; sizes whose scratch need (fa_decode_workspace_bytes) exceeds
 *     FA_DECODE_STATIC_SCRATCH_BYTES are rejected with FA_ERR_TOO_LARGE and
 *     nothing is enqueued.  FA_ERR_TOO_LARGE comes only after every check
 *     that fa_decode makes before touching the device (sizes, scale,
 *     pointers, overlaps) has passed.
 *   - The first call on a device looks up the device address of the scratch
 *     array (cudaGetSymbolAddress, with that device current; a failure is
 *     returned as FA_ERR_CUDA), which may load the library's device code.  Make
 *     that first call on each device before any stream capture begins.
 *   - There is one scratch array per device.  Calls that may run at the same
 *     time on one device (other streams, other host threads) overwrite each
 *     other's partial results: order them, e.g. on one stream.
 *   - Nothing in the scratch needs to start at zero: each call writes every
 *     partial result before reading it.
 */
#define FA_DECODE_STATIC_SCRATCH_BYTES (8u << 20)
fa_status fa_decode_static(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal,
                           float scale, fa_stream_t stream);

/*
 * fa_bwd_workspace_bytes — device scratch that fa_bwd needs for these sizes:
 * B*H*Np*(Dp + 2)*4 bytes, Np = N rounded up to a multiple of 64 and Dp the
 * padded head size (64 for d <= 64, else 128): the per-row L*log2 e and D,
 * and the fp32 dQ accumulator, kept at the padded head size.  Needs no
 * device.  Errors: FA_ERR_INVALID_ARG (bytes NULL, sizes < 1 or too large),
 * FA_ERR_UNSUPPORTED (d not a multiple of 8 in 8..128).  B*H must not exceed
 * 65535.
 */
fa_status fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, size_t *bytes);

/*
 * fa_bwd — gradients of fa_fwd's attention with respect to q, k and v for
 * the output gradient dout ("Writing and Benchmarking Custom Kernels"
 * §10.3.2, backward-pass recomputation): the probabilities are recomputed
 * tile by tile from the forward's logsumexp, never stored.  For each (b, h),
 * with P the attention probabilities of fa_fwd and L its logsumexp:
 *     D_i   = dO_i . O_i
 *     dV_j  = sum_i P_ij dO_i
 *     dS_ij = P_ij (dO_i . V_j - D_i)
 *     dQ_i  = scale * sum_j dS_ij K_j,   dK_j = scale * sum_i dS_ij Q_i
 * (sums over the pairs the mask lets through: j <= i when causal).
 *
 * Arguments
 *   q, k, v    device pointers, bf16, contiguous (B, H, N, d): the forward's inputs.
 *   o, lse     the forward's outputs for those inputs (o bf16 (B, H, N, d),
 *              lse fp32 (B, H, N), natural log); same causal and scale.
 *   dout       device pointer, bf16, contiguous (B, H, N, d): dLoss/dO.
 *   dq, dk, dv device pointers, bf16, contiguous (B, H, N, d); fully written.
 *   B, H       B*H <= 65535.  d: a multiple of 8 from 8 to 128 (as fa_fwd).
 *              causal: 0 or 1.  scale: finite, > 0
 *              (the forward's).
 *   workspace, workspace_bytes
 *              device scratch of at least fa_bwd_workspace_bytes(...) bytes,
 *              16-byte aligned; nothing in it needs to start at zero.  Calls
 *              that may run at the same time must not share it.
 *   stream     CUDA stream the three kernels (prepare, main, dQ convert) are
 *              enqueued on.
 *
 * Ownership: the caller owns every buffer; the library allocates nothing.
 * Bf16 pointers and the workspace 16-byte aligned, lse 4-byte aligned,
 * else FA_ERR_UNSUPPORTED.  Outputs and workspace may overlap no input and
 * no other output (FA_ERR_INVALID_ARG).  Asynchrony, FA_ERR_CUDA and
 * FA_ERR_TIMEOUT reporting as for fa_fwd.  dQ is accumulated in fp32 in the
 * workspace: each step adds its contribution with one bulk tensor reduce-add
 * (cp.reduce.async.bulk.tensor, the add done in L2) per block of 64 query
 * rows and 32 head dims.  The order of those adds depends on timing, so the
 * last bits of dQ may differ between runs; dK and dV are deterministic.
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t H, int64_t N,
                 int64_t d, int causal, float scale, void *workspace, size_t workspace_bytes,
                 fa_stream_t stream);

/*
 * fa_bias_gelu_dropout — the fused elementwise chain of "Fusion and IO-aware
 * kernels" (§ The idea in one minute: a bias add, a GELU and a dropout, one
 * HBM read and one HBM write instead of three round trips), with the tanh
 * form of GELU of "Writing and Benchmarking Custom Kernels" §10.2.1.  For
 * element (r, c), flat index e = r*cols + c:
 *     h = x[r][c] + bias[c]
 *     g = 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3)))
 *     y[r][c] = g / (1 - p) if bit e % 32 of keep[e / 32] is set, else 0
 *
 * Arguments
 *   x        device pointer, bf16, contiguous (rows, cols).
 *   bias     device pointer, bf16, (cols).
 *   keep     device pointer, uint32 words of keep bits over the flat index
 *            (ceil(rows*cols / 32) words; the dropout's random draws, made by
 *            the caller), or NULL to keep every element.
 *   y        device pointer, bf16, contiguous (rows, cols); fully written.
 *   rows, cols  >= 1; cols a multiple of 8 (else FA_ERR_UNSUPPORTED).
 *   p        dropout probability, 0 <= p < 1; kept values are scaled by 1/(1-p).
 *   stream   CUDA stream the one launch is enqueued on.
 *
 * Ownership: the caller owns every buffer.  x, bias, y 16-byte aligned and
 * keep 4-byte aligned, else FA_ERR_UNSUPPORTED.  y may not overlap x, bias or
 * keep (FA_ERR_INVALID_ARG); x may be y's input only out of place.
 * Asynchrony, launch and FA_ERR_CUDA as for fa_fwd.
 */
fa_status fa_bias_gelu_dropout(const void *x, const void *bias, const uint32_t *keep, void *y,
                               int64_t rows, int64_t cols, float p, fa_stream_t stream);

/*
 * fa_check_device_status — synchronises `stream`, reads and clears the
 * device-side status word of the current device.  Returns FA_ERR_TIMEOUT if a
 * kernel launched since the last check gave up a bounded wait (its outputs are
 * then incomplete), FA_ERR_CUDA if the copy or synchronisation failed or a
 * kernel refused to run (shared memory not 1024-byte aligned), FA_OK
 * otherwise.  `where`, if not NULL, receives the code of the first wait that
 * gave up (0 if none).
 *
 * The status word is per device, not per stream: it collects the reports of
 * every kernel of this library on the device, whatever stream launched it,
 * and the check waits only for `stream`.  Kernels still running on other
 * streams may report after the read; the clear removes only the bits that
 * were read (an atomic update on the device), so such a later report stays
 * for the next check.
 */
fa_status fa_check_device_status(fa_stream_t stream, uint32_t *where);

/*
 * fa_get_device_status — fa_check_device_status without the wait code:
 * synchronises `stream`, reads and clears the device status word of the
 * current device, and returns FA_OK, FA_ERR_TIMEOUT (a kernel gave up a
 * bounded wait; its outputs are incomplete) or FA_ERR_CUDA.  The deferred
 * report of errors that happen inside a launch ("Writing and Benchmarking
 * Custom Kernels" §10.2.1: kernel errors surface only at a later
 * synchronisation).
 */
fa_status fa_get_device_status(fa_stream_t stream);

/*
 * fa_set_wait_limit_ns — upper bound, in nanoseconds, on any single pipeline
 * wait inside the kernels launched after this call (default 1e9 = 1 s; 0
 * restores the default).  Affects only how quickly a stuck kernel gives up.
 */
fa_status fa_set_wait_limit_ns(uint64_t ns);

/*
 * fa_debug_skip_k_tile — test hook for the failure path.  With tile >= 0, the
 * first CTA of every later fa_fwd launch never loads its tile-th K tile, and
 * that of every later fa_bwd launch never loads the Q / dout tile of its
 * tile-th step, so the MMA warp's wait for it runs out after the wait limit,
 * the kernel abandons its work and fa_check_device_status reports
 * FA_ERR_TIMEOUT; no fault, trap or hang is involved.  -1 (the default) turns
 * it off.  Outputs of a launch made with the hook on are incomplete.
 */
fa_status fa_debug_skip_k_tile(int tile);

/*
 * fa_debug_set_schedule — test hook for the forward's causal item order.
 * The persistent forward kernel takes its causal work items either in pairs
 * (a heavy and a light query block of one head, which keeps that head's K
 * and V in L2) or in cost order (heaviest first, snaking over the CTAs),
 * and chooses by size: cost order when all heads' K and V fit in 60% of L2.
 * order = 0 forces the pair order and 1 the cost order on every later
 * causal fa_fwd launch (non-causal launches have one order only); -1 (the
 * default) restores the choice by size.  Both orders compute every row the
 * same way, so the results are identical to the bit; only the speed
 * differs.  FA_ERR_INVALID_ARG for any other value.
 */
fa_status fa_debug_set_schedule(int order);

/*
 * fa_debug_decode_plan — test hook: the split plan fa_decode would use for
 * these sizes if `wave` CTAs of its partial kernel were resident at once (on
 * a device, wave = resident CTAs per SM x SMs).  Host arithmetic only: no
 * device call.  Writes the number of chunks the key range is cut into
 * (*splits; 1 = not split) and the keys per chunk (*chunk, the last chunk
 * may be shorter).  The plan weighs a whole number of waves of equal chunks
 * against the partial results that splitting adds.
 * FA_ERR_INVALID_ARG for null outputs, wave < 1 or sizes fa_decode refuses
 * as invalid; FA_ERR_UNSUPPORTED as fa_decode reports it.
 */
fa_status fa_debug_decode_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t wave,
                               int *splits, int *chunk);

/* Static description of a status code (never NULL). */
const char *fa_status_string(fa_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
