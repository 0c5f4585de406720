// kernels.h -- host-side launchers of the qmm kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/qmm.h"

namespace qmm {

cudaError_t launch_dequant(int dtype, const void *w, float *out, int64_t m, int64_t k, int64_t rb, float ts,
                           int num_sms, cudaStream_t st);

// Small-batch GEMV (1 <= n <= 8).  status: device status word; limit_ns:
// the bound on every wait inside the kernel.
cudaError_t launch_gemv(int dtype, const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k,
                        int n, int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st);

// The split-K register-X GEMV for Q4_0/Q8_0/Q4_K/Q6_K/NVFP4 when it has a plan
// for the problem; cudaErrorNotSupported (nothing launched) otherwise.
cudaError_t launch_gemv_sk(int dtype, const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k,
                           int n, int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st);

// MoE gate/up GEMV over 2 * n_pairs matrices; tokens = rows of x.
cudaError_t launch_moe_gemv(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const float *x,
                            float *y, int64_t in_f, int64_t n_ff, int n_used, int n_pairs, int tokens, int num_sms,
                            uint32_t *status, uint64_t limit_ns, cudaStream_t st);

// MoE down projection: y[t][gin] = the fixed-order sum (u = 0, 1, ...) of
// token t's n_used pair products of gin rows over n_ff -- in one grouped
// register-X launch when a token's pairs fit its k teams (part unused),
// else per-pair products into part [n_pairs][gin] (into y directly when
// n_used == 1) and the combine kernel.
cudaError_t launch_moe_down(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const float *h,
                            float *y, float *part, int64_t n_ff, int64_t gin, int n_used, int tokens, int num_sms,
                            uint32_t *status, uint64_t limit_ns, cudaStream_t st);

// y[t][gin] = the fixed-order sum (u = 0, 1, ...) of part[t*n_used + u][gin].
cudaError_t launch_moe_combine(const float *part, float *y, int64_t gin, int n_used, int tokens, int num_sms,
                               cudaStream_t st);

// Q8_1 activation blocks: q[rows][k] int8, d[rows][k/32] (k % 32 == 0).
cudaError_t launch_quantize_q8_1(const float *x, int8_t *q, float *d, int64_t rows, int64_t k, int num_sms,
                                 cudaStream_t st);

// NVFP4 (36-byte groups or V2 rows) MoE products on Q8_1 activations:
// dst[mat][r] = scales[mat] * sum_c W_mat[r][c] * q[a][c] * d[a][c/32] with
// activation row a = (mat % n_pairs) / n_used, for mats matrices of
// rows_per_mat rows; k % 64 == 0, k <= QMM_Q8_MAX_K.
// With x non-null the kernel quantizes the activation rows x [act rows][k]
// float32 itself (the same bytes launch_quantize_q8_1 writes; q, d unused).
cudaError_t launch_moe_q8(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const int8_t *q,
                          const float *d, const float *x, float *dst, int64_t k, int64_t rows_per_mat, int mats,
                          int n_pairs, int n_used, int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st);

// Activation rows [rows][k] f32 -> NVFP4 V2 rows (E2M1 codes, one E4M3 scale
// per 16, nearest values, decided in float32); k % 256 == 0.
cudaError_t launch_quantize_nvfp4(const float *x, void *out, int64_t rows, int64_t k, int num_sms, cudaStream_t st);

// dst[n][m] = sum_k W[m][k] Xq[n][k], W and Xq NVFP4 V2 rows, on the
// block-scaled FP4 tensor cores; k % 256 == 0.
cudaError_t launch_gemm_fp4(const void *w, const void *xq, float *dst, int64_t m, int64_t k, int64_t n, int num_sms,
                            uint32_t *status, uint64_t limit_ns, cudaStream_t st);
cudaError_t gemm_fp4_init();

// NVFP4 36-byte-group rows -> V2 rows (codes, then the scale stream); k % 64 == 0.
cudaError_t launch_nvfp4_repack_v2(const uint8_t *v1, uint8_t *v2, int64_t m, int64_t k, int num_sms,
                                   cudaStream_t st);

// Tensor-core GEMM for n > QMM_GEMV_MAX_N.  x16 is the f16 workspace (packed
// formats only).  status: the handle's device status word.
struct GemmArgs {
    int dtype;
    const void *w;
    int64_t rb;
    const float *x;
    float *dst;
    int64_t m, k, n;
    void *x16;
    uint32_t *status;
    uint64_t wait_limit_ns;
    int debug_skip_first_b_load;  // test hook: leave one stage unloaded so a wait runs out
};
cudaError_t launch_gemm_tc(const GemmArgs &a, int num_sms, cudaStream_t st);
cudaError_t gemm_tc_init();

}  // namespace qmm
