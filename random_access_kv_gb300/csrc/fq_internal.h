// Internal declarations shared by the translation units of libfq.so.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/fq.h"

struct fq_ctx {
    int device;
    int d, k, N, B, nb, R;      // nb = d / k blocks, B = log2 N, R = nb * B
    float *C;                    // [N x k] codebook
    float *cc;                   // [N] |c_n|^2
    float *Pi;                   // [d x d] rotation, row-major
    float *Crot;                 // k == d: [N x d] rotated codebook C Pi (row n = Pi^T c_n)
    uint32_t *flags;             // [0] sticky FQ_FLAG_* word, [1] the copy fq_status takes
    int num_sms;
    // k = 2 tensor-core encoder tables
    uint8_t *pi_split;           // fp16 halves of 2^12 Pi, swizzled as the MMA's B operand
    uint32_t *grid2;             // candidate grid and overflow slots
    float g_scale, g_offs;       // grid cell of u: round(u * g_scale + g_offs)
    int k2_max_ctas;             // co-resident CTAs of the k = 2 encoder
    // tensor-core decoder tables
    uint8_t *pit_split;          // fp16 halves of 2^12 Pi^T, swizzled as the MMA's B operand
    uint16_t *cb_split;          // [N][2k] fp16 halves of 2^10 c_n (k hi, then k lo)
    uint32_t *cb_lanes;          // d = 64, k <= 2: cb_split's words, each repeated for 32 lanes
    // k = d tensor-core encoder table
    uint16_t *crot_split;        // fp16 halves of -2 * 2^12 Crot (hi block [N x d], lo block), then bf16 norm blocks
    // k = 4 candidate-grid encoder tables
    uint16_t *k4_cells;          // [G^4][8] cell records (count, up to 7 ascending indices)
    uint16_t *k4_pool;           // overflow lists of cells with more than 7 candidates
    uint8_t *k4_axis;            // lattice entry -> coarse cell index per axis (0xFF outside)
    float *k4_ncb;               // [N x 4] negated codebook
    float k4_fs;                 // lattice entries per unit of a coordinate
    int k4_G, k4_max_ctas;
    // k = 4, 8 tensor-core encoder table
    uint8_t *cb_ops;             // codebook rows as MMA B operands (see fq_encode_kq.cu)
    int kq_max_ctas;
    int smem_optin;              // dynamic shared memory a CTA may opt in to
    // fused attention launch plans: [0] one query per cluster, [1] four queries of one group
    // (nwarps == 0: the plan does not fit)
    struct AttendPlan {
        int qg, lut, nwarps, max_split;
        int64_t slots[9];        // co-resident CTAs per cluster size
        size_t smem;
    } attend[2];
};

namespace fq {

using AttendPlan = fq_ctx::AttendPlan;

// Mapping from an input row r to its store row: (r / n_new) * seq_cap + row_base + r % n_new.
// fq_encode uses n_new = M (one sequence) and row_base = row0.
struct RowMap {
    int64_t n_new;
    int64_t seq_cap;
    int64_t row_base;
    __host__ __device__ __forceinline__ int64_t operator()(int64_t r) const {
        int64_t s = r / n_new;
        return s * seq_cap + row_base + (r - s * n_new);
    }
};

// Kernel launchers (defined in the .cu files). Each returns a cudaError_t from the launch.
cudaError_t launch_encode_blocks(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map,
                                 float *nu, uint32_t *codes, cudaStream_t s);
cudaError_t launch_decode_blocks(const fq_ctx *ctx, const float *nu, const uint32_t *codes,
                                 int64_t M, const int64_t *idx, int64_t n, void *out,
                                 bool out_f32, cudaStream_t s);
cudaError_t launch_encode_full(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map,
                               float *nu, uint32_t *codes, cudaStream_t s);
cudaError_t launch_decode_full(const fq_ctx *ctx, const float *nu, const uint32_t *codes,
                               int64_t M, const int64_t *idx, int64_t n, void *out,
                               bool out_f32, cudaStream_t s);
// Tensor map of a row-major fp16 [M x D] matrix in 128-row x 64-column boxes, 128-byte swizzle.
bool encode_rows_tensor_map(CUtensorMap *tm, const void *x, int64_t M, int D);
// fp16 hi/lo halves of scale * src (d x d, row n = MMA row n) in the K-major 128-byte swizzle layout.
void split_operand_sw128(const float *src, int d, float scale, std::vector<uint16_t> &out);

bool k2_tc_supported(const fq_ctx *ctx);
cudaError_t prepare_k2_tc(fq_ctx *ctx);
cudaError_t launch_encode_k2_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                uint32_t *codes, cudaStream_t s);
bool decode_tc_supported(const fq_ctx *ctx);
cudaError_t prepare_decode_tc(fq_ctx *ctx);
cudaError_t launch_decode_tc(const fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                             const int64_t *idx, int64_t n, void *out, bool out_f32, cudaStream_t s);
bool full_tc_supported(const fq_ctx *ctx);
cudaError_t prepare_full_tc(fq_ctx *ctx);
cudaError_t launch_encode_full_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                  uint32_t *codes, cudaStream_t s);
bool k4_grid_supported(const fq_ctx *ctx);
cudaError_t prepare_k4_grid(fq_ctx *ctx);
cudaError_t launch_encode_k4_grid(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                  uint32_t *codes, cudaStream_t s);
bool kq_tc_supported(const fq_ctx *ctx);
cudaError_t prepare_kq_tc(fq_ctx *ctx);
cudaError_t launch_encode_kq_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                uint32_t *codes, cudaStream_t s);
cudaError_t launch_centroid_sums(const fq_ctx *ctx, const __half *x, int64_t M, const float *nu,
                                 const uint32_t *codes, double *sums, double *counts, cudaStream_t s);
cudaError_t launch_wait_selftest(const fq_ctx *ctx, uint64_t limit_ns, cudaStream_t s);
// flags[1] = atomic exchange of flags[0] with 0, by one device thread: a read-and-clear of the
// sticky word that loses no flag raised meanwhile by a kernel on another stream.
cudaError_t launch_take_flags(uint32_t *flags, cudaStream_t s);
cudaError_t prepare_attend(fq_ctx *ctx);
cudaError_t launch_attend(const fq_ctx *ctx, const float *nu, const uint32_t *codes, const __half *q,
                          int64_t n_queries, int64_t q_per_group, int64_t T, int64_t k_row0, int64_t v_row0,
                          int64_t stride, float scale, float *out, cudaStream_t s);
bool attend_supported(const fq_ctx *ctx);
// One-time kernel attribute set-up (dynamic shared memory limits); called by fq_codebook_load.
cudaError_t prepare_encode_blocks(const fq_ctx *ctx);
cudaError_t prepare_decode_blocks(const fq_ctx *ctx);
cudaError_t prepare_full(const fq_ctx *ctx);

}  // namespace fq
