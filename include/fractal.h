/*
 * fractal.h - C ABI of the iterated-map archive of symbol streams (part of libfq.so), sm_103a.
 *
 * The archive is the storage primitive of the page "Fractal KV-Cache Archives" (gist.science
 * summary of arXiv 2607.07144), cited below as [Archive §x]. It stores the index stream a vector
 * quantiser produces (for instance FibQuant's codeword indices) as points of the plane:
 *   [Archive §Method 1, mechanism] a regular N-gon with vertex V(c) = (cos 2 pi c/N, sin 2 pi c/N)
 *       per symbol c; symbol c_k maps the current point by p_k = V(c_k) + r (p_{k-1} - V(c_k));
 *   [Archive §Method 1, properties] the map is lossless when r keeps the symbols' cells (discs of
 *       radius r about (1 - r) V(c)) disjoint, i.e. r < sin(pi/N) / (1 + sin(pi/N)); encoding is
 *       linear; a position is read back from the nearest stored anchor;
 *   [Archive §Method 1, implementation] one point (the anchor) is stored per segment of L symbols,
 *       and a segment is rebuilt from its anchor by a backward search: the symbol is the cell that
 *       holds the point, then that symbol's map is inverted.
 * Readings of what the page leaves open: every segment starts at the origin (segments are
 * independent); forward steps are computed in fp64 per coordinate as t = p - V, p = r t + V (one
 * fused multiply-add), always in that order, so anchors do not depend on how segments are split
 * across calls.
 *
 * Layout. A batch of n_streams streams of capacity T_cap symbols keeps S_cap = ceil(T_cap / L)
 * anchors per stream: anchors is double [n_streams][S_cap][2] (x, y), 16-byte aligned, stream q's
 * segment s at index q S_cap + s. Segment s holds positions [s L, s L + L) of its stream; the last
 * one may be partial. Symbols are uint16_t. All streams of a batch hold the same number T of
 * symbols (they advance together, as the (layer, head) streams of a KV cache do).
 *
 * Conventions are those of fq.h: caller-owned device buffers, asynchronous calls on a stream
 * (void* cudaStream_t, NULL = legacy default stream) that validate on the host and return FQ_*
 * codes (fq.h), the current device left as it was, one host thread per context. Conditions only
 * the device can see set sticky bits that fa_status() reads and clears.
 */
#ifndef FQ_FRACTAL_H
#define FQ_FRACTAL_H

#include <stdint.h>

#include "fq.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fa_ctx fa_ctx;

/* Sticky device flags returned by fa_status(). */
enum {
    FA_FLAG_SYMBOL = 1u,   /* an appended symbol was >= N: its segment's anchor is set to NaN */
    FA_FLAG_RANGE = 2u,    /* an fa_access position was outside the batch: its output is 0xFFFF */
    FA_FLAG_CORRUPT = 4u   /* a backward step met a point outside every cell (an anchor that no
                              encode of these parameters wrote): those symbols are 0xFFFF */
};

/* sin(pi/N) / (1 + sin(pi/N)): contraction ratios strictly below it give disjoint cells. 0 if N < 2. */
double fa_ratio_limit(int N);

/*
 * fa_max_segment - the longest segment whose backward search is exact in fp64 for (N, r), capped
 * at 64; 0 if r is not in (0, fa_ratio_limit(N)) or not one symbol fits.
 * Bound used: a forward step's rounding error per coordinate is below 1.01 u (1 + 4 r) (that of a
 * rounded product and a rounded sum; the fused form this library uses errs less) and a
 * backward step's below 8 u (u = 2^-53); the error of the rebuilt point grows by 1/r per backward
 * step, and all L decisions of a segment are correct when it stays below half the margin
 * (1 - r) sin(pi/N) - r between a cell and the edges of its angular sector.
 */
int fa_max_segment(int N, double r);

/*
 * fa_create - a context for alphabet size N, contraction ratio r and segment length L on `device`.
 *   N : 2 <= N <= 4096.
 *   r : 0 < r < fa_ratio_limit(N), with a cell margin of at least 2e-5 (the backward search decides
 *       cells in fp32 and needs that room).
 *   L : 1 <= L <= fa_max_segment(N, r).
 * The vertex table V [N][2] is computed here on the host in double precision (cos and sin of
 * 2 pi c / N) and copied to the device with the fp32 cell centres (1 - r) V(c). Blocking.
 * Returns FQ_OK and *out, or FQ_EINVAL / FQ_ENOMEM / FQ_ECUDA / FQ_ENODEV and *out = NULL.
 */
int fa_create(fa_ctx **out, int N, double r, int L, int device);

/* fa_params - the context's N, r and L (any pointer may be NULL). */
int fa_params(const fa_ctx *ctx, int *N, double *r, int *L);

/* fa_vertex_table - copies the vertex table, double [N][2], to host memory V_host. Blocking. */
int fa_vertex_table(const fa_ctx *ctx, double *V_host);

/* fa_segments - anchors per stream of capacity T_cap: ceil(T_cap / L); -1 on bad arguments (T_cap < 1 or
 * within 64 of INT64_MAX). */
int64_t fa_segments(const fa_ctx *ctx, int64_t T_cap);

/*
 * fa_encode - append n_new symbols to every stream of a batch that holds T_old symbols per stream
 * [Archive §Method 1: linear-time encode, O(1) append]. T_old = 0 encodes streams from scratch.
 *   sym     : device uint16_t [n_streams][n_new], stream q's new symbols in order.
 *   anchors : device double [n_streams][S_cap][2], S_cap = fa_segments(ctx, T_cap). Updated in
 *             place: a partial last segment continues from its stored point, later segments start
 *             at the origin; untouched anchors are not written.
 * Requires T_old >= 0, n_new >= 0, T_old + n_new <= T_cap. One device thread per touched segment.
 * The resulting anchors are bit-identical whatever the split of the stream into calls.
 */
int fa_encode(fa_ctx *ctx, const uint16_t *sym, int64_t n_streams, int64_t n_new, int64_t T_cap,
              int64_t T_old, double *anchors, void *stream);

/*
 * fa_decode - every symbol of every stream: out device uint16_t [n_streams][T] (row pitch T).
 * One device thread per segment, backward from its anchor [Archive §Method 1, anchored backward
 * search]. 0 <= T <= T_cap.
 */
int fa_decode(fa_ctx *ctx, const double *anchors, int64_t n_streams, int64_t T_cap, int64_t T,
              uint16_t *out, void *stream);

/*
 * fa_access - random access [Archive §Method 1, random access from the nearest anchor]: out[i] =
 * the symbol at flat position pos[i] = q T_cap + t (stream q, position t < T), rebuilt backward
 * from segment t / L's anchor down to t only (at most L steps). pos is device int64_t [n]; out is
 * device uint16_t [n]. A position outside the batch gives 0xFFFF and FA_FLAG_RANGE.
 */
int fa_access(fa_ctx *ctx, const double *anchors, int64_t n_streams, int64_t T_cap, int64_t T,
              const int64_t *pos, int64_t n, uint16_t *out, void *stream);

/* fa_status - reads and clears the context's sticky FA_FLAG_* bits in one atomic exchange on the device
 * (as fq_status), then synchronises `stream`. */
int fa_status(fa_ctx *ctx, void *stream, uint32_t *flags);

/* fa_destroy - frees the context's device tables. NULL is a no-op. */
void fa_destroy(fa_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* FQ_FRACTAL_H */
