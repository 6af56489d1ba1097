/*
 * fq.h - C ABI of the FibQuant codec library (libfq.so), GB300 / sm_103a.
 *
 * The codec is the one described on the page "FibQuant: universal vector quantisation for
 * random-access KV-cache compression" (gist.science summary of arXiv 2605.11478), cited below
 * as [FibQuant §x]:
 *   encoder [FibQuant §2.3]: nu = ||x||_2, u = Pi x / nu, split u into d/k blocks of size k,
 *            index of the nearest codeword of a shared codebook C [N x k] for every block;
 *   storage [FibQuant §1, §2.3]: every vector's d/k indices (B = log2 N bits each) at a fixed
 *            bit address, R = (d/k) B bits per vector, rate b = log2(N)/k bits per coordinate;
 *   decoder [FibQuant §2.3]: fetch the codewords, concatenate, apply Pi^T, scale by nu.
 *
 * Conventions shared by every call:
 *   - Every device buffer is allocated and owned by the caller. The library never frees or
 *     keeps a caller pointer beyond the call.
 *   - Every call that takes a stream (a cudaStream_t passed as void*, NULL = legacy default
 *     stream) is asynchronous: it validates its arguments on the host, enqueues kernels and
 *     returns. Invalid arguments return an error code and enqueue nothing.
 *   - Conditions only the device can see (a gather index outside [0, M), a non-finite input
 *     element, a bounded wait that gave up) set sticky bits of a per-context device flag word
 *     instead of faulting; fq_status() reads and clears them. Such rows are written as zeros.
 *   - The calling thread's current device is left as it was.
 *   - A context is not thread-safe: calls on one context must come from one host thread at a
 *     time. Calls on different contexts are independent.
 *
 * Bit layout of the codes: a little-endian stream of uint32 words. Vector m's record occupies
 * stream bits [m R, m R + R), bit i of the stream being bit (i mod 32) of word i / 32. Block
 * b's index occupies record bits [b B, b B + B), least significant bit first. There is no
 * padding between records, so the rate is exactly b bits per coordinate. A buffer for M
 * vectors holds fq_code_words(ctx, M) words.
 */
#ifndef FQ_H
#define FQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fq_ctx fq_ctx;

/* Return codes. */
enum {
    FQ_OK = 0,
    FQ_EINVAL = 1,   /* bad argument: null pointer, bad size, unsupported (d, k, N), non-finite table */
    FQ_ENOMEM = 2,   /* device or host allocation failed (fq_codebook_load only) */
    FQ_ECUDA = 3,    /* a CUDA runtime call or kernel launch failed */
    FQ_EALIGN = 4,   /* a buffer is not aligned as the call requires */
    FQ_ENODEV = 5    /* no CUDA device, or the device is not sm_103 */
};

/* Sticky device flags returned by fq_status(). */
enum {
    FQ_FLAG_RANGE = 1u,      /* a gather index was outside [0, M): that output row is zero */
    FQ_FLAG_NONFINITE = 2u,  /* an input vector had a NaN or Inf: its codes are 0 and nu = 0 */
    FQ_FLAG_TIMEOUT = 4u     /* a bounded device-side wait gave up: that tile's output is invalid */
};

/*
 * fq_codebook_load - build a context holding the shared codebook and rotation on `device`.
 *   C_host  : host float32 [N x k], row n = codeword c_n [FibQuant §2.2]. Copied.
 *   N       : codebook size, a power of two, 2 <= N <= 65536.
 *   k       : block size. Supported: k in {1, 2, 4, 8} with d in {64, 128}; k in {1, 2, 3, 4, 8}
 *             with d = 96 (CUDA-core kernels only; k = 3 takes the Fibonacci-sphere codebook of
 *             [FibQuant §2.2]); and k = d = 64.
 *   Pi_host : host float32 [d x d], row-major, the shared rotation u = Pi x [FibQuant §2.1].
 *             Used as given (orthogonality is the caller's business). Copied.
 *   d       : vector dimension (head dim).
 *   device  : CUDA device ordinal.
 * Derived tables built here, on the host in double precision: |c_n|^2, the rotated codebook
 * C Pi for k = d, and the split half-precision copies of Pi used by the tensor-core rotation.
 * Returns FQ_OK and *out, or an error and *out = NULL. The caller keeps ownership of the host
 * arrays. Blocking (copies complete before return). With FQ_TEST_FAIL_ALLOC set in the
 * environment its device allocations fail, so that the FQ_ENOMEM path can be tested.
 */
int fq_codebook_load(fq_ctx **out, const float *C_host, int N, int k,
                     const float *Pi_host, int d, int device);

/*
 * fq_encode - encode M vectors [FibQuant §2.3, encoder] into rows row0 .. row0+M-1 of a code
 * store.
 *   x     : device fp16 [M x d], row-major, 16-byte aligned.
 *   nu    : device float32 [row0 + M], receives nu_m = ||x_m||_2 at index row0 + m. 4-byte aligned.
 *   codes : device uint32 code store; the records of rows row0 .. row0+M-1 are written, every
 *           other bit of the store is left unchanged (boundary words are updated with atomic
 *           masked writes). 4-byte aligned, at least fq_code_words(ctx, row0 + M) words.
 *   row0  : first destination row (>= 0), e.g. the current cache length when appending.
 * A zero vector gets nu = 0 and all-zero indices.
 */
int fq_encode(fq_ctx *ctx, const void *x, int64_t M, float *nu, uint32_t *codes,
              int64_t row0, void *stream);

/*
 * fq_encode_append - streaming append into n_seq independent sequences (e.g. one per layer
 * and head), each with capacity seq_capacity rows, of n_new new vectors each at positions
 * t0 .. t0+n_new-1. Input row s*n_new + i goes to store row s*seq_capacity + t0 + i.
 *   x : device fp16 [n_seq x n_new x d]; nu, codes: as fq_encode, sized for n_seq*seq_capacity rows.
 * Requires t0 + n_new <= seq_capacity. Same encoder as fq_encode [FibQuant §2.3].
 */
int fq_encode_append(fq_ctx *ctx, const void *x, int64_t n_seq, int64_t n_new,
                     int64_t seq_capacity, int64_t t0, float *nu, uint32_t *codes,
                     void *stream);

/*
 * fq_decode - decode all M rows of a code store [FibQuant §2.3, decoder]:
 * x_hat_m = nu_m Pi^T concat_b(c_{i_mb}), written as fp16 (round to nearest even).
 *   nu    : device float32 [M];  codes : device uint32 store of M records;
 *   out   : device fp16 [M x d], 16-byte aligned.
 */
int fq_decode(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M, void *out,
              void *stream);

/*
 * fq_decode_gather - random-access decode [FibQuant §1: any token decodes on its own by address
 * arithmetic; §2.3 decoder]: out row j = decode of store row idx[j].
 *   nu, codes : the store of M rows (as fq_decode);
 *   idx       : device int64 [n], row indices; an index outside [0, M) writes a zero row and
 *               sets FQ_FLAG_RANGE.
 *   out       : device fp16 [n x d], 16-byte aligned.
 */
int fq_decode_gather(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                     const int64_t *idx, int64_t n, void *out, void *stream);

/*
 * fq_decode_gather_f32 - as fq_decode_gather but writes the float32 value before the final
 * fp16 rounding (out: device float32 [n x d], 16-byte aligned). For accuracy checks.
 */
int fq_decode_gather_f32(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                         const int64_t *idx, int64_t n, float *out, void *stream);

/*
 * fq_attend - single-query softmax attention over compressed keys and values, decoded inside the
 * kernel [FibQuant §5: the fixed-address interface lets decompression fuse into attention; §2.3
 * decoder]. For query r (group g = r / q_per_group):
 *   o_r = sum_t p_t x_hat(v_row0 + g stride + t) / sum_t p_t,
 *   p_t = exp(s_t - max_t s_t),  s_t = scale * q_r . x_hat(k_row0 + g stride + t),  t < T,
 * where x_hat(m) is the decode of store row m (as fq_decode, before fp16 rounding).
 *   nu, codes   : the store of M rows (keys and values of all groups in one store);
 *   q           : device fp16 [n_queries x d], row-major;
 *   n_queries   : a multiple of q_per_group (queries sharing one cached group, >= 1);
 *   T           : cached tokens per group, >= 1;
 *   k_row0, v_row0, stride : row of key/value token t of group g is row0 + g * stride + t; every
 *                 such row must lie in [0, M) (else FQ_EINVAL);
 *   scale       : finite score scale (commonly 1/sqrt(d));
 *   out         : device float32 [n_queries x d].
 * Non-finite norms in the store give non-finite outputs. Returns FQ_EINVAL for d = 96 contexts
 * (no attention kernel) and when the codebook and record staging of this context do not fit one
 * CTA's shared memory.
 */
int fq_attend(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M, const void *q,
              int64_t n_queries, int64_t q_per_group, int64_t T, int64_t k_row0, int64_t v_row0,
              int64_t stride, float scale, float *out, void *stream);

/*
 * fq_centroid_sums - the centroid step of a Lloyd iteration on the codebook [FibQuant §2.2,
 * refinement: Lloyd iterations on draws of the block source minimise the finite codebook's MSE].
 * The assignment step is fq_encode of the training rows; this call then adds, for every codeword n,
 *   sums[n][0..k) += sum of the blocks u_b (u = Pi x / nu) whose index is n,
 *   counts[n]     += their number,
 * over rows m < M. Rows with nu = 0 are skipped.
 *   x      : device fp16 [M x d], the encoded rows, 16-byte aligned;
 *   nu, codes : the store fq_encode wrote for exactly these rows (row m at record m);
 *   sums   : device float64 [N x k], counts : device float64 [N], accumulated (the caller zeroes).
 * The new codebook is sums[n] / counts[n] wherever counts[n] > 0.
 */
int fq_centroid_sums(fq_ctx *ctx, const void *x, int64_t M, const float *nu, const uint32_t *codes,
                     double *sums, double *counts, void *stream);

/*
 * fq_selftest_wait - exercise the failure path of the kernels' bounded waits: a kernel waits on
 * a barrier that nothing completes, gives up after about limit_ns nanoseconds (at most 1e9) and
 * sets FQ_FLAG_TIMEOUT, which the next fq_status reports. Nothing traps; the context stays usable.
 * (The codec itself has no counterpart; the method's pages describe no failure handling.)
 */
int fq_selftest_wait(fq_ctx *ctx, uint64_t limit_ns, void *stream);

/* Number of uint32 words of a store of M records: ceil(M R / 32), R = (d/k) log2 N bits per record
 * at a fixed address per vector [FibQuant §1 fixed address; §2.3 rate]. Returns -1 on bad arguments. */
int64_t fq_code_words(const fq_ctx *ctx, int64_t M);

/* R = (d/k) log2 N, bits per record [FibQuant §2.3, rate]. Returns -1 for a NULL context. */
int fq_record_bits(const fq_ctx *ctx);

/* d, k and N of a context (any output pointer may be NULL): head dimension, block size and codebook
 * size of [FibQuant §2.3, encoder]. Returns FQ_EINVAL for a NULL context. */
int fq_shape(const fq_ctx *ctx, int *d, int *k, int *N);

/*
 * fq_status - read and clear the context's sticky device flags (FQ_FLAG_*) into *flags, then
 * synchronise `stream`. The read-and-clear is one atomic exchange on the device, ordered after the
 * work already queued on `stream`; a flag raised at the same time by a kernel on another stream is
 * either returned now or kept for the next call, never lost. Returns FQ_ECUDA if the stream reports
 * an error. (Failure reporting of this library; the method's pages describe none.)
 */
int fq_status(fq_ctx *ctx, void *stream, uint32_t *flags);

/* Free a context and its device tables. Synchronises the context's device. NULL is a no-op. */
void fq_destroy(fq_ctx *ctx);

/* Static, human-readable text of a return code. */
const char *fq_strerror(int err);

#ifdef __cplusplus
}
#endif

#endif /* FQ_H */
