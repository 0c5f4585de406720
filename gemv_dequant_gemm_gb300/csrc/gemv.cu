// gemv.cu -- the small-batch GEMV (1 <= n <= 8) and the MoE gate/up GEMV.
//
// dst[i][row] = sum_c W[row][c] * X[i][c] read straight from the packed
// weights at their packed size, as the batched GEMV described in
// aprender-serve 0.70.2 cublas_prefill/mod.rs does (doc comment of
// cublas_gemm_threshold, which also names that GEMV's one-warp blocks as its
// weakness; this kernel spreads every row over a whole CTA instead).
//
// A CTA owns R consecutive rows.  All of its threads split the row's k range
// into 8-weight groups (thread t takes groups t, t+T, ...), so consecutive
// threads read consecutive bytes of each row.  The X values of a group are
// loaded once and reused for the R rows; each weight is decoded once
// (decode8, float32, exact) and used for the n activation rows.  Partial sums
// are reduced by warp shuffles and then across warps in a fixed order, so the
// result is deterministic.  Every group's 8 products are summed into a fresh
// partial before joining the accumulator, which keeps the float32 rounding
// error far below 1e-5 * sum|W*X|.
//
// The MoE kernel (memra-engine 0.128.0 moe_rows_ceiling_bench.rs, the served
// gate/up kernel over ptrs[plane*n_pairs + j]) is the same body with n = 1:
// grid.y walks the 2*n_pairs (plane, pair) matrices, each CTA multiplies its
// rows of one matrix by the pair's token and scales by scales[matrix].
#include "decode.cuh"
#include "kernels.h"

namespace qmm {

__device__ __forceinline__ void load8_x(const float *xrow, int64_t e0, int64_t k, bool vec_ok, float (&v)[8]) {
    if (vec_ok && e0 + 8 <= k) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(xrow + e0));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(xrow + e0) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (e0 + j < k) ? __ldg(xrow + e0 + j) : 0.0f;
    }
}

template <int F>
__device__ __forceinline__ void decode_group(const uint8_t *row, int64_t e0, int64_t k, float (&w)[8]) {
    if constexpr (F == QMM_F32) {
        decode8_f32(row, e0, k, w);
    } else {
        constexpr int QK = Fmt<F>::QK, BB = Fmt<F>::BB;
        decode8<F>(row + (e0 / QK) * BB, static_cast<int>(e0 % QK), 1.0f, w);
    }
}

// Shared body: rows [r0, r0 + R) of W (row stride rb, `rows` valid from r0),
// NV activation rows of x (row stride k).  Returns in red[] (thread 0..R*NV-1
// read it after the final barrier) the per-(row, i) sums.
template <int F, int NV, int R, int T>
__device__ __forceinline__ void gemv_body(const uint8_t *__restrict__ w, int64_t rb, const float *__restrict__ x,
                                          int64_t k, int rows, float *red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t ngroups = (k + 7) / 8;
    const bool vec_ok = (k % 4) == 0;
    float acc[R][NV];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[r][i] = 0.0f;

    for (int64_t g = tid; g < ngroups; g += T) {
        const int64_t e0 = g * 8;
        float xv[NV][8];
#pragma unroll
        for (int i = 0; i < NV; ++i) load8_x(x + i * k, e0, k, vec_ok, xv[i]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < rows) {
                float wv[8];
                decode_group<F>(w + r * rb, e0, k, wv);
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    float part = wv[0] * xv[i][0];
#pragma unroll
                    for (int j = 1; j < 8; ++j) part = __fmaf_rn(wv[j], xv[i][j], part);
                    acc[r][i] += part;
                }
            }
        }
    }
    constexpr int NW = T / 32;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float v = acc[r][i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane == 0) red[warp * (R * NV) + r * NV + i] = v;
        }
    __syncthreads();
    if (tid < R * NV) {
        float s = red[tid];
#pragma unroll
        for (int wi = 1; wi < NW; ++wi) s += red[wi * (R * NV) + tid];
        red[tid] = s;
    }
    __syncthreads();
}

template <int F, int NV, int R, int T>
__global__ void __launch_bounds__(T) gemv_kernel(const uint8_t *__restrict__ w, int64_t rb,
                                                 const float *__restrict__ x, float *__restrict__ dst, int64_t m,
                                                 int64_t k) {
    __shared__ float red[(T / 32) * R * NV];
    griddep_wait();
    griddep_launch();
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R;
    const int rows = static_cast<int>(m - r0 < R ? m - r0 : R);
    gemv_body<F, NV, R, T>(w + r0 * rb, rb, x, k, rows, red);
    const int tid = threadIdx.x;
    if (tid < R * NV) {
        const int r = tid / NV, i = tid % NV;
        if (r < rows) dst[static_cast<int64_t>(i) * m + r0 + r] = red[tid];
    }
}

template <int F, int R, int T>
__global__ void __launch_bounds__(T) moe_gemv_kernel(const void *const *__restrict__ w_ptrs, int64_t rb,
                                                     const float *__restrict__ scales, const float *__restrict__ x,
                                                     float *__restrict__ y, int64_t in_f, int64_t n_ff, int n_used,
                                                     int n_pairs, uint32_t *status) {
    __shared__ float red[(T / 32) * R];
    griddep_wait();
    griddep_launch();
    const int mat = blockIdx.y;
    const int pair = mat % n_pairs;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R;
    const int rows = static_cast<int>(n_ff - r0 < R ? n_ff - r0 : R);
    const uint8_t *wm = static_cast<const uint8_t *>(w_ptrs[mat]);
    if (wm == nullptr || (reinterpret_cast<uintptr_t>(wm) & 15u) != 0) {
        // a bad table entry: report it and leave this matrix's rows as NaN
        if (threadIdx.x == 0) atomicOr(status, kDevBadPtr);
        if (threadIdx.x < rows) y[static_cast<int64_t>(mat) * n_ff + r0 + threadIdx.x] = __int_as_float(0x7FC00000);
        return;
    }
    gemv_body<F, 1, R, T>(wm + r0 * rb, rb, x + static_cast<int64_t>(pair / n_used) * in_f, in_f, rows, red);
    const int tid = threadIdx.x;
    if (tid < rows) y[static_cast<int64_t>(mat) * n_ff + r0 + tid] = __ldg(scales + mat) * red[tid];
}

template <int F, int NV>
static cudaError_t launch_gemv_nv(const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k,
                                  cudaStream_t st) {
    constexpr int R = NV <= 2 ? 4 : 8;
    const auto *wb = static_cast<const uint8_t *>(w);
    const unsigned grid = static_cast<unsigned>((m + R - 1) / R);
    if ((k + 7) / 8 <= 128)
        return launch_pdl(gemv_kernel<F, NV, R, 128>, dim3(grid), dim3(128), 0, st, 1u, wb, rb, x, dst, m, k);
    return launch_pdl(gemv_kernel<F, NV, R, 256>, dim3(grid), dim3(256), 0, st, 1u, wb, rb, x, dst, m, k);
}

template <int F>
static cudaError_t launch_gemv_f(const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k, int n,
                                 cudaStream_t st) {
    switch (n) {
    case 1: return launch_gemv_nv<F, 1>(w, rb, x, dst, m, k, st);
    case 2: return launch_gemv_nv<F, 2>(w, rb, x, dst, m, k, st);
    case 3: return launch_gemv_nv<F, 3>(w, rb, x, dst, m, k, st);
    case 4: return launch_gemv_nv<F, 4>(w, rb, x, dst, m, k, st);
    case 5: return launch_gemv_nv<F, 5>(w, rb, x, dst, m, k, st);
    case 6: return launch_gemv_nv<F, 6>(w, rb, x, dst, m, k, st);
    case 7: return launch_gemv_nv<F, 7>(w, rb, x, dst, m, k, st);
    case 8: return launch_gemv_nv<F, 8>(w, rb, x, dst, m, k, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(int dtype, const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k, int n,
                        int /*num_sms*/, cudaStream_t st) {
    switch (dtype) {
    case QMM_F32: return launch_gemv_f<QMM_F32>(w, rb, x, dst, m, k, n, st);
    case QMM_Q4_0: return launch_gemv_f<QMM_Q4_0>(w, rb, x, dst, m, k, n, st);
    case QMM_Q8_0: return launch_gemv_f<QMM_Q8_0>(w, rb, x, dst, m, k, n, st);
    case QMM_Q4_K: return launch_gemv_f<QMM_Q4_K>(w, rb, x, dst, m, k, n, st);
    case QMM_Q6_K: return launch_gemv_f<QMM_Q6_K>(w, rb, x, dst, m, k, n, st);
    case QMM_NVFP4: return launch_gemv_f<QMM_NVFP4>(w, rb, x, dst, m, k, n, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int F>
static cudaError_t launch_moe_f(const void *const *w_ptrs, int64_t rb, const float *scales, const float *x, float *y,
                                int64_t in_f, int64_t n_ff, int n_used, int n_pairs, uint32_t *status,
                                cudaStream_t st) {
    constexpr int R = 4;
    const dim3 grid(static_cast<unsigned>((n_ff + R - 1) / R), static_cast<unsigned>(2 * n_pairs));
    if ((in_f + 7) / 8 <= 128)
        return launch_pdl(moe_gemv_kernel<F, R, 128>, grid, dim3(128), 0, st, 1u, w_ptrs, rb, scales, x, y, in_f, n_ff,
                          n_used, n_pairs, status);
    return launch_pdl(moe_gemv_kernel<F, R, 256>, grid, dim3(256), 0, st, 1u, w_ptrs, rb, scales, x, y, in_f, n_ff,
                      n_used, n_pairs, status);
}

cudaError_t launch_moe_gemv(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const float *x,
                            float *y, int64_t in_f, int64_t n_ff, int n_used, int n_pairs, uint32_t *status,
                            cudaStream_t st) {
    switch (dtype) {
    case QMM_F32: return launch_moe_f<QMM_F32>(w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, status, st);
    case QMM_Q4_0: return launch_moe_f<QMM_Q4_0>(w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, status, st);
    case QMM_Q8_0: return launch_moe_f<QMM_Q8_0>(w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, status, st);
    case QMM_Q4_K: return launch_moe_f<QMM_Q4_K>(w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, status, st);
    case QMM_Q6_K: return launch_moe_f<QMM_Q6_K>(w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, status, st);
    case QMM_NVFP4: return launch_moe_f<QMM_NVFP4>(w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, status, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
