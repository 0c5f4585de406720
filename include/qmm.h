/*
 * qmm.h -- C ABI of the GB300 (sm_103a) quantized-weight projection matmul.
 *
 * The operation is the projection matmul of an LLM layer,
 *
 *     dst[n][m] = sum_k W[m][k] * X[n][k],
 *
 * the matmul that cera 0.4.0 examples/wgpu_gemm_bench.rs benchmarks (doc
 * comment of struct Shape: src0 is [m][k], src1 is [n][k], dst is [n][m]),
 * where W is kept in a packed block-quantized format and decoded inside the
 * kernels.
 *
 * Layouts (all row-major, all dense, no padding between rows):
 *   W    [m][k] packed: each row is k/QK consecutive blocks of BB bytes
 *        (qmm_row_bytes), rows back to back.  f32 weights are plain floats.
 *   X    [n][k] float32, row stride k.
 *   dst  [n][m] float32, row stride m (m contiguous, as in that page's
 *        comparison comment on its output stride).
 *
 * Block formats (QK weights per block / BB bytes per block), packed sizes as in
 * the VARIANTS table of the same page and the NVFP4 groups of memra-engine
 * 0.128.0 src/bin/moe_rows_ceiling_bench.rs, synth_rows:
 *   QMM_F32    1 / 4     IEEE float32
 *   QMM_Q4_0   32 / 18   f16 d; 16 bytes, low nibble of byte j = element j,
 *                        high nibble = element j+16; value (q-8)*d
 *   QMM_Q8_0   32 / 34   f16 d; 32 int8; value q*d
 *   QMM_Q4_K  256 / 144  f16 d, f16 dmin, 12 bytes of 6-bit scales/mins for 8
 *                        sub-blocks of 32, 128 bytes of nibbles;
 *                        value d*sc*q - dmin*min
 *   QMM_Q6_K  256 / 210  128 bytes low 4 bits, 64 bytes high 2 bits, 16 int8
 *                        scales (16 weights each), f16 d; value d*sc*(q-32)
 *   QMM_NVFP4  64 / 36   4 E4M3 scale bytes (one per 16 weights), 32 bytes of
 *                        E2M1 codes, low nibble of byte j = element 2j;
 *                        value e2m1*e4m3
 *   QMM_NVFP4_V2 32 / 18 the same values with the scales split out: a row is
 *                        its k/2 code bytes (low nibble of byte j = element
 *                        2j), then its k/16 E4M3 scale bytes (byte s covers
 *                        elements 16s..16s+15); 18 bytes per 32 weights as in
 *                        the V2 arms of memra-engine 0.128.0
 *                        moe_rows_ceiling_bench.rs (main), built from
 *                        QMM_NVFP4 rows by qmm_nvfp4_repack_v2.  The calls
 *                        take it with k % 64 == 0 (aligned code words), in
 *                        qmm_gemv, qmm_moe_gemv, qmm_moe_down and qmm_dequant;
 *                        qmm_gemm and qmm_gemm_noalloc with n > QMM_GEMV_MAX_N
 *                        return QMM_ERR_UNSUPPORTED for it.
 * The bit orders inside Q4_K and Q6_K are the ggml k-quant orders.
 *
 * Conventions shared by every call:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never frees, keeps or reallocates them.  The handle owns only a 4-byte
 *     device status word allocated by qmm_create.
 *   - Pointers must be 16-byte aligned (any cudaMalloc / torch allocation is).
 *     Packed weight buffers must stay readable up to the next 16-byte boundary
 *     after their last byte (true of every cudaMalloc allocation).
 *   - Calls are asynchronous on the caller's stream (a cudaStream_t passed as
 *     void*, NULL = the legacy default stream).  The return value reports the
 *     host-side checks and the launch; errors found on the device (a bounded
 *     wait that expired) are latched in the handle and returned by
 *     qmm_sync_status.
 *   - No call allocates device memory after qmm_create, so every call can be
 *     issued while a stream is being captured into a CUDA graph.
 *   - Outputs are fully overwritten and are a deterministic function of the
 *     inputs (no atomics in the arithmetic): two identical calls give
 *     bit-identical results.
 *   - Output buffers must not overlap any input buffer.
 *   - There is no CPU fallback: without an sm_103 device every compute call
 *     returns an error.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qmm_ctx *qmm_handle;

typedef enum {
    QMM_F32 = 0,
    QMM_Q4_0 = 1,
    QMM_Q8_0 = 2,
    QMM_Q4_K = 3,
    QMM_Q6_K = 4,
    QMM_NVFP4 = 5,
    QMM_NVFP4_V2 = 6
} qmm_dtype;

/* Status codes. */
enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1, /* null pointer or handle, unknown dtype       */
    QMM_ERR_UNSUPPORTED = 2, /* dtype not supported by this call            */
    QMM_ERR_SHAPE = 3,       /* size out of range or k not a whole block    */
    QMM_ERR_ALIGN = 4,       /* pointer not 16-byte aligned                 */
    QMM_ERR_ARCH = 5,        /* device is not sm_103 (GB300)                */
    QMM_ERR_CUDA = 6,        /* a CUDA runtime call failed                  */
    QMM_ERR_TIMEOUT = 7,     /* a device-side bounded wait expired          */
    QMM_ERR_WORKSPACE = 8,   /* workspace missing or too small              */
    QMM_ERR_OVERLAP = 9      /* an output overlaps an input                 */
};

/* Largest n that qmm_gemv accepts; qmm_gemm sends n <= this to the same
 * kernel (the small-batch regime, cf. the GEMM-vs-GEMV threshold of
 * aprender-serve 0.70.2 cublas_prefill/mod.rs, cublas_gemm_threshold). */
#define QMM_GEMV_MAX_N 8

/* Create a handle on CUDA device `device`.  Checks that the device is sm_103,
 * allocates the 4-byte device status word.  *out is set on success only.
 * Errors: QMM_ERR_INVALID_ARG (out == NULL), QMM_ERR_ARCH, QMM_ERR_CUDA. */
int qmm_create(int device, qmm_handle *out);

/* Free the handle and its status word.  Waits for nothing: the caller must
 * not destroy a handle with calls still running.  NULL is accepted. */
int qmm_destroy(qmm_handle h);

/* Static description of a status code; never NULL. */
const char *qmm_strerror(int status);

/* QK (weights per block) and BB (bytes per block) of a dtype; 0 if unknown. */
int64_t qmm_block_weights(qmm_dtype t);
int64_t qmm_block_bytes(qmm_dtype t);

/* Bytes of one packed row of k weights, k/QK*BB; 0 if k is not a positive
 * whole number of blocks or t is unknown.  Host-only, needs no device. */
int64_t qmm_row_bytes(qmm_dtype t, int64_t k);

/* Device workspace, in bytes, that qmm_gemm needs for this problem (0 when it
 * needs none: n <= QMM_GEMV_MAX_N, or f32 weights).  For the packed formats
 * at n > QMM_GEMV_MAX_N it holds the f16 copy of X that the tensor-core
 * kernel reads: n*k*2 bytes rounded up to 256.  Host-only. */
size_t qmm_gemm_workspace_bytes(qmm_dtype t, int64_t m, int64_t k, int64_t n);

/* dst[n][m] = sum_k W[m][k] * X[n][k]  (cera wgpu_gemm_bench.rs, struct
 * Shape; the prefill GEMM of its 512-token LFM2 shapes).
 *   n <= QMM_GEMV_MAX_N: the fp32-FMA GEMV kernel (same as qmm_gemv).
 *   n >  QMM_GEMV_MAX_N: the tensor-core kernel: packed W is decoded to f16 in
 *     shared memory, X is rounded to f16 (round to nearest even) into the
 *     workspace, products accumulate in fp32 in tensor memory (tcgen05
 *     kind::f16).  f32 W uses kind::tf32 on X and W as given.  Decoded weights
 *     and X must lie within the f16 range on this path.
 * Accuracy: |dst - exact| <= 2e-3 * sum_k |W*X| + 1e-6 per element on the
 * tensor-core path, 1e-5 * sum_k |W*X| on the GEMV path.
 * Sizes: 1 <= m, n <= 2^24; 1 <= k <= 2^20 and k % QK == 0.  workspace must be
 * a device buffer of at least qmm_gemm_workspace_bytes(...) bytes (may be NULL
 * when that is 0).  Errors: QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE,
 * QMM_ERR_ALIGN, QMM_ERR_WORKSPACE, QMM_ERR_OVERLAP, QMM_ERR_CUDA. */
int qmm_gemm(qmm_handle h, qmm_dtype t, const void *w, const float *x, float *dst, int64_t m,
             int64_t k, int64_t n, void *workspace, size_t workspace_bytes, void *stream);

/* The small-batch GEMV: the same product for 1 <= n <= QMM_GEMV_MAX_N, read
 * straight from the packed weights at their packed size, as the batched
 * GEMV of aprender-serve 0.70.2 cublas_prefill/mod.rs does (doc comment of
 * cublas_gemm_threshold).  fp32 decode and fp32 FMA; accuracy
 * |dst - exact| <= 1e-5 * sum_k |W*X|.  All dtypes.  Errors as qmm_gemm, and
 * QMM_ERR_SHAPE for n outside 1..QMM_GEMV_MAX_N. */
int qmm_gemv(qmm_handle h, qmm_dtype t, const void *w, const float *x, float *dst, int64_t m,
             int64_t k, int64_t n, void *stream);

/* MoE gate/up GEMV over routed experts (memra-engine 0.128.0
 * src/bin/moe_rows_ceiling_bench.rs: the served gate/up kernel, its pointer
 * table ptrs[plane*n_pairs + j] and its per-matrix scales scl[pr]).
 * With n_pairs = t_tokens * n_used, for plane p in {0 = gate, 1 = up} and
 * pair j < n_pairs (token j / n_used):
 *   y[p][j][r] = scales[p*n_pairs + j] * sum_c W_pj[r][c] * x[j / n_used][c]
 * for r < n_ff, where W_pj = w_ptrs[p*n_pairs + j] is an [n_ff][in_f] packed
 * matrix.  w_ptrs is a DEVICE array of at least 2*n_pairs device pointers
 * (the page's 3*n_pairs table, whose third plane holds down projections, is
 * accepted as is; entries past 2*n_pairs are not read).  scales is a device
 * float array of at least 2*n_pairs entries, x is [t_tokens][in_f] float32,
 * y is [2][n_pairs][n_ff] float32.  The activation stays fp32 (no int8
 * re-quantization) and no clamp or gating is applied.  Any dtype; every
 * matrix pointer must be 16-byte aligned.  Accuracy as qmm_gemv, relative to
 * |scale| * sum_c |W*x|.  Sizes: 1 <= n_used, t_tokens; n_pairs <= 4096;
 * 1 <= n_ff <= 2^24; in_f % QK == 0.  Errors as qmm_gemv. */
int qmm_moe_gemv(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                 const float *x, float *y, int64_t in_f, int64_t n_ff, int n_used, int t_tokens,
                 void *stream);

/* MoE down projection over routed experts (memra-engine 0.128.0
 * src/bin/moe_rows_ceiling_bench.rs: the down step after gate/up, one
 * [gin][n_ff] matrix per pair at ptrs[2*n_pairs + j] of that page's table,
 * the pairs of a token accumulated into y).  With n_pairs = t_tokens * n_used
 * and pair j = i*n_used + u of token i:
 *   y[i][r] = sum over u < n_used of scales[j] * sum_c W_j[r][c] * hact[j][c]
 * for r < gin, where W_j = w_ptrs[j] is a [gin][n_ff] packed matrix and
 * hact[j] is that pair's n_ff activations (the gated gate/up output).
 *   - w_ptrs: DEVICE array of n_pairs device pointers (pass table + 2*n_pairs
 *     for a gate/up/down table laid out as that page's), each 16-byte
 *     aligned; a NULL or misaligned entry makes its token's rows NaN and
 *     latches QMM_ERR_ALIGN for qmm_sync_status.
 *   - scales: device float[n_pairs], the factor of each pair (its routing
 *     weight, a per-matrix scale, or their product: the call only multiplies).
 *   - hact: device float32 [n_pairs][n_ff]; y: device float32 [t_tokens][gin],
 *     overwritten (not accumulated into).
 *   - workspace: device scratch of qmm_moe_down_workspace_bytes(gin, n_used,
 *     t_tokens) bytes (0 when n_used == 1: then pass NULL), 16-byte aligned,
 *     overlapping no other argument, any contents.  When n_ff >= 2048 and
 *     n_used divides 512 so that
 *     teams of 512/n_used threads cover n_ff in whole blocks (16 weights
 *     for NVFP4, 8 otherwise) with at most 32 values per thread -- at
 *     n_ff = 2048: n_used 4 or 8 for NVFP4, 2, 4 or 8 for the others -- one
 *     kernel takes each token's pairs together and sums them itself,
 *     leaving the workspace unused; otherwise the workspace holds the
 *     per-pair products and a second kernel sums them.  Either way each
 *     token's pairs are added in the order u = 0, 1, ... so results are
 *     deterministic.
 * Any dtype; fp32 decode and FMA; accuracy |y - exact| <= 1e-5 *
 * sum_u |scales[j]| * sum_c |W_j * hact_j|.  Sizes: 1 <= n_used, t_tokens;
 * n_pairs <= 4096; 1 <= gin <= 2^24; n_ff % QK == 0.  Errors as qmm_moe_gemv,
 * and QMM_ERR_WORKSPACE (workspace missing or too small). */
size_t qmm_moe_down_workspace_bytes(int64_t gin, int n_used, int t_tokens);
int qmm_moe_down(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                 const float *hact, float *y, int64_t n_ff, int64_t gin, int n_used, int t_tokens,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Largest row length (in_f of qmm_moe_gemv_q8, n_ff of qmm_moe_down_q8) the
 * int8-activation calls accept. */
#define QMM_Q8_MAX_K 8192

/* Q8_1 activation blocks (memra-engine 0.128.0
 * src/bin/moe_rows_ceiling_bench.rs, main: quantize_q8_1 turns the f32
 * activation into int8 codes with per-block scales before its served gate/up
 * kernel; the page prints neither its code nor its rule).  For every block of
 * 32 consecutive values of a row of x ([rows][k] float32, k % 32 == 0):
 *   d = amax / 127,  q = x * (1/d) rounded to the nearest integer, halves away
 *   from zero (q = 0 when d == 0),
 * each step one float32 operation, so the integer codes are decided in
 * float32 and match any IEEE float32 implementation of the same steps bit for
 * bit.  q is [rows][k] int8, d is [rows][k/32] float32.  Device pointers, all
 * 16-byte aligned, outputs overlapping no input; 1 <= rows <= 2^24, 32 <= k <=
 * 2^20.  Errors: QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE, QMM_ERR_ALIGN,
 * QMM_ERR_OVERLAP, QMM_ERR_CUDA. */
int qmm_quantize_q8_1(qmm_handle h, const float *x, int8_t *q, float *d, int64_t rows, int64_t k,
                      void *stream);

/* qmm_moe_gemv on Q8_1 activations (the same page's served gate/up kernel
 * reads the quantized activation and names its PRMT/dp4a instruction stream):
 *   y[p][j][r] = scales[p*n_pairs + j] * sum_c W_pj[r][c] * q[i][c] * d[i][c/32]
 * with i = j / n_used, the token of pair j; q [t_tokens][in_f] int8 and d
 * [t_tokens][in_f/32] float32 as qmm_quantize_q8_1 writes them.  NVFP4 and
 * NVFP4_V2 weights only (QMM_ERR_UNSUPPORTED otherwise): each 16-weight
 * region's product is an exact int32 dot product of 2*e2m1 codes and q,
 * scaled once by its E4M3 scale and block scale d.  Accuracy |y - exact| <=
 * 1e-5 * |scale| * sum_c |W * q*d| against the exact product on the quantized
 * activation.  in_f % 64 == 0, in_f <= QMM_Q8_MAX_K; other sizes, pointer
 * table, scales and y as qmm_moe_gemv; q, d 16-byte aligned.  The 7.0
 * argument of the page's kernel (its meaning is not printed) is not applied.
 * Errors as qmm_moe_gemv. */
int qmm_moe_gemv_q8(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                    const int8_t *q, const float *d, float *y, int64_t in_f, int64_t n_ff, int n_used,
                    int t_tokens, void *stream);

/* qmm_moe_down on Q8_1 activations: hact[j][c] is given as q[j][c] *
 * d[j][c/32] (q [n_pairs][n_ff] int8, d [n_pairs][n_ff/32] float32).  The
 * same products, workspace and fixed-order combine as qmm_moe_down, with the
 * arithmetic of qmm_moe_gemv_q8; NVFP4 and NVFP4_V2 only; n_ff % 64 == 0,
 * n_ff <= QMM_Q8_MAX_K.  Accuracy |y - exact| <= 1e-5 * sum_u |scales[j]| *
 * sum_c |W_j * q*d|.  Workspace: qmm_moe_down_workspace_bytes(gin, n_used,
 * t_tokens).  Errors as qmm_moe_down. */
int qmm_moe_down_q8(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                    const int8_t *q, const float *d, float *y, int64_t n_ff, int64_t gin, int n_used,
                    int t_tokens, void *workspace, size_t workspace_bytes, void *stream);

/* The two calls above with the quantization inside the product kernel: x is
 * the float32 activation (qmm_moe_gemv_q8_fused: [t_tokens][in_f], one row
 * per token; qmm_moe_down_q8_fused: [n_pairs][n_ff], one row per pair),
 * 16-byte aligned, overlapping neither y nor the workspace.  Each CTA turns
 * the activation values its lanes multiply into Q8_1 codes and block scales
 * with the steps of qmm_quantize_q8_1, so y is bit-identical to
 * qmm_quantize_q8_1 followed by qmm_moe_gemv_q8 / qmm_moe_down_q8 on the same
 * x; one kernel launch fewer, and no q, d buffers.  Other arguments, limits,
 * accuracy and errors as those calls. */
int qmm_moe_gemv_q8_fused(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                          const float *x, float *y, int64_t in_f, int64_t n_ff, int n_used, int t_tokens,
                          void *stream);
int qmm_moe_down_q8_fused(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                          const float *x, float *y, int64_t n_ff, int64_t gin, int n_used, int t_tokens,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Activation rows for the block-scaled FP4 product (qmm_gemm_fp4): x
 * [rows][k] float32 becomes NVFP4 V2 rows xq (rows * qmm_row_bytes(
 * QMM_NVFP4_V2, k) bytes: k/2 code bytes, element 2j in the low nibble of
 * byte j, then k/16 E4M3 scale bytes).  Per block of 16 consecutive values:
 * scale = the E4M3 value nearest amax/6, code = the E2M1 value nearest
 * x/scale, ties to the even code, both saturating at the format's largest
 * finite value (448, 6); zero codes when the scale is zero.  Every step is a
 * float32 operation, so the bytes match any IEEE implementation of the same
 * steps.  The pages fix no activation rule for an FP4 tensor-core product
 * (memra-engine 0.128.0 moe_rows_ceiling_bench.rs keeps its weights in NVFP4
 * and quantizes its activation to Q8_1; aprender-serve 0.70.2
 * cublas_prefill/mod.rs names an FP8 activation scratch for its low-precision
 * GEMM): this is the plainest reading, the activation in the weights' own
 * NVFP4 groups.  Useful range: |x| <= 2688 (6 * 448); blocks whose amax/6 is
 * below 2^-10 quantize to zero.  1 <= rows <= 2^24, 256 <= k <= 2^20, k % 256
 * == 0; device pointers, 16-byte aligned, not overlapping.  Errors:
 * QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE, QMM_ERR_ALIGN, QMM_ERR_OVERLAP,
 * QMM_ERR_CUDA. */
int qmm_quantize_nvfp4(qmm_handle h, const float *x, void *xq, int64_t rows, int64_t k, void *stream);

/* The prefill product on the block-scaled FP4 tensor cores (tcgen05
 * kind::mxf4nvf4): dst[n][m] = sum_k W[m][k] * Xq[n][k] with W [m][k] and Xq
 * [n][k] both NVFP4 V2 rows (weights repacked from 36-byte groups by
 * qmm_nvfp4_repack_v2, activations written by qmm_quantize_nvfp4).  Each
 * product of two E2M1 values and each 16-term block sum is exact; the block
 * sums are scaled by the two E4M3 scales and accumulated in fp32.  Accuracy
 * |dst - exact| <= 2e-3 * sum_k |W * Xq| + 1e-6 against the exact product on
 * the quantized activation (the tensor-core tolerance).  1 <= m, n <= 2^24,
 * 256 <= k <= 2^20, k % 256 == 0; device pointers, 16-byte aligned, dst
 * overlapping neither input.  Errors: QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE,
 * QMM_ERR_ALIGN, QMM_ERR_OVERLAP, QMM_ERR_CUDA; device-side timeouts through
 * qmm_sync_status. */
int qmm_gemm_fp4(qmm_handle h, const void *w, const void *xq, float *dst, int64_t m, int64_t k, int64_t n,
                 void *stream);

/* Repack NVFP4 rows into the V2 layout (memra-engine 0.128.0
 * src/bin/moe_rows_ceiling_bench.rs, main: the V2 arms read the same values
 * through rows repacked with the scales split out).  v1 is [m] rows of
 * k/64 * 36 bytes (QMM_NVFP4), v2 receives [m] rows of k/32 * 18 bytes
 * (QMM_NVFP4_V2): for every row, 64-weight group g's 32 code bytes go to
 * bytes 32g..32g+31 of the row and its 4 scale bytes to bytes k/2 + 4g ..
 * k/2 + 4g + 3.  A pure byte permutation: every weight keeps its value.
 * Device pointers, both 16-byte aligned and not overlapping; 1 <= m <= 2^24,
 * 64 <= k <= 2^20, k % 64 == 0.  Errors: QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE,
 * QMM_ERR_ALIGN, QMM_ERR_OVERLAP, QMM_ERR_CUDA. */
int qmm_nvfp4_repack_v2(qmm_handle h, const void *v1, void *v2, int64_t m, int64_t k, void *stream);

/* Standalone dequant (aprender-serve cublas_prefill/mod.rs module doc, v1
 * path, which dequantizes Q4K/Q6K weights into an FP32 scratch buffer):
 * out[m][k] float32 = the decoded
 * value of W[m][k], rounded once to float32; for QMM_NVFP4 the decoded value
 * times tensor_scale, rounded once (pass 1.0f otherwise; it is ignored for the
 * other dtypes).  Bit-exact with the formats' definitions.  Sizes as qmm_gemm
 * (m*k <= 2^40).  Errors: QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE, QMM_ERR_ALIGN,
 * QMM_ERR_OVERLAP, QMM_ERR_CUDA. */
int qmm_dequant(qmm_handle h, qmm_dtype t, const void *w, float *out, int64_t m, int64_t k,
                float tensor_scale, void *stream);

/* Synchronize `stream`, then return and clear the device status latched by
 * earlier calls on this handle: QMM_OK; QMM_ERR_TIMEOUT (a bounded wait ran
 * out; that call's output is not valid); QMM_ERR_ALIGN (a qmm_moe_gemv table
 * entry was NULL or not 16-byte aligned; its rows were set to NaN); or
 * QMM_ERR_CUDA if the synchronization itself failed. */
int qmm_sync_status(qmm_handle h, void *stream);

/* Size of the scratch area that qmm_gemm_noalloc uses: 8 MiB. */
#define QMM_NOALLOC_SCRATCH_BYTES (8u << 20)

/* qmm_gemm for callers that cannot allocate device memory: code that runs
 * where cudaMalloc is unavailable or forbidden (inside a custom allocator or
 * a memory-pool callback, in a process whose device memory is fully handed
 * out to another framework, or under a policy that bans allocation after
 * start-up).  It needs neither a handle (qmm_create allocates a status word)
 * nor a caller workspace: the f16 copy of X that the tensor-core kernel reads
 * lives in a static device array of QMM_NOALLOC_SCRATCH_BYTES built into the
 * library.  The paper pages have no counterpart of this call.
 *   - Same product, layouts, accuracy and size rules as qmm_gemm, on the
 *     current device; n <= QMM_GEMV_MAX_N goes to the GEMV kernel as there.
 *   - n * k * 2 must not exceed QMM_NOALLOC_SCRATCH_BYTES - 256 when
 *     n > QMM_GEMV_MAX_N and the weights are packed; larger problems return
 *     QMM_ERR_WORKSPACE.
 *   - When the memory is taken: under CUDA's lazy module loading (the
 *     default, CUDA_MODULE_LOADING=LAZY) the driver places the scratch array
 *     and each kernel on a device the first time they are used there, not
 *     when the library is loaded.  So the first call on a device (of this
 *     function or of qmm_gemm_noalloc_status) takes the array's memory, and
 *     the first call that runs a given kernel (tensor-core or GEMV path, per
 *     dtype) loads that kernel's code.  Callers that cannot allocate later
 *     should make those calls at start-up, or set CUDA_MODULE_LOADING=EAGER
 *     before CUDA initializes, which places everything when the context is
 *     created.  After that, calls allocate nothing.
 *   - The first call on a device also sets that device up (looks up the
 *     array's device address, checks the architecture, sets kernel
 *     attributes); make it before any stream capture.  A set-up that fails
 *     is retried by the next call.
 *   - Every call shares the one scratch array, whose contents persist from
 *     call to call: calls that overlap on the GPU (on different streams, or
 *     from different threads) race on it.  Serialize them.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.  Device-side wait timeouts are latched in the scratch array's
 *     status word; read them with qmm_gemm_noalloc_status.
 * Errors: QMM_ERR_INVALID_ARG, QMM_ERR_SHAPE, QMM_ERR_ALIGN,
 * QMM_ERR_OVERLAP, QMM_ERR_WORKSPACE, QMM_ERR_UNSUPPORTED, QMM_ERR_ARCH,
 * QMM_ERR_CUDA. */
int qmm_gemm_noalloc(qmm_dtype t, const void *w, const float *x, float *dst, int64_t m, int64_t k,
                     int64_t n, void *stream);

/* The device status latched by qmm_gemm_noalloc calls on the current device
 * since the last read: synchronizes `stream`, copies the status word into a
 * host variable, clears it and returns QMM_OK, QMM_ERR_TIMEOUT (a bounded
 * wait ran out; the output of a call since the last read is not valid) or
 * QMM_ERR_CUDA.  Allocates nothing.  It sets the device up like the first
 * qmm_gemm_noalloc call, so a caller can also use it at start-up for that.
 * The paper pages have no counterpart of this call. */
int qmm_gemm_noalloc_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
