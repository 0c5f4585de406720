// api.cu -- the extern "C" entry points declared in include/qmm.h:
// handle life cycle, host-side argument checks, regime dispatch (GEMV for
// n <= QMM_GEMV_MAX_N, tensor cores above), device status read-back.
#include <stdint.h>
#include <stdlib.h>

#include "../../include/qmm.h"
#include "../../include/qmm_testing.h"
#include "kernels.h"

struct qmm_ctx {
    uint32_t magic;
    int device;
    int num_sms;
    uint32_t *d_status;      // device status word (kDev* bits)
    uint64_t wait_limit_ns;  // bound of every device-side wait
    int debug_skip_first_b_load;
};

namespace {

constexpr uint32_t kMagic = 0x716D6D31u;  // "qmm1"
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
constexpr int64_t kMaxMN = int64_t(1) << 24;
constexpr int64_t kMaxK = int64_t(1) << 20;

bool valid_handle(qmm_handle h) { return h != nullptr && h->magic == kMagic; }

bool known_dtype(int t) { return t >= QMM_F32 && t <= QMM_NVFP4_V2; }

// k is a whole number of blocks; V2 rows also need k % 64 == 0, which keeps
// every 4-byte code word of every row aligned.
bool k_ok(qmm_dtype t, int64_t k) {
    return qmm_row_bytes(t, k) != 0 && (t != QMM_NVFP4_V2 || k % 64 == 0);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Runs `fn` with the handle's device current, restoring the caller's device.
template <typename Fn> int on_device(qmm_handle h, Fn fn) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return QMM_ERR_CUDA;
    if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return QMM_ERR_CUDA;
    const cudaError_t e = fn();
    if (prev != h->device) cudaSetDevice(prev);
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

// Checks shared by the product calls.
int check_product(qmm_handle h, qmm_dtype t, const void *w, const float *x, const float *dst, int64_t m, int64_t k,
                  int64_t n) {
    if (!valid_handle(h) || !known_dtype(t) || !w || !x || !dst) return QMM_ERR_INVALID_ARG;
    if (m < 1 || n < 1 || m > kMaxMN || n > kMaxMN || k < 1 || k > kMaxK) return QMM_ERR_SHAPE;
    if (!k_ok(t, k)) return QMM_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(x) || !aligned16(dst)) return QMM_ERR_ALIGN;
    const size_t wbytes = static_cast<size_t>(qmm_row_bytes(t, k) * m);
    const size_t dbytes = static_cast<size_t>(n * m) * sizeof(float);
    if (overlaps(dst, dbytes, w, wbytes) || overlaps(dst, dbytes, x, static_cast<size_t>(n * k) * sizeof(float)))
        return QMM_ERR_OVERLAP;
    return QMM_OK;
}

}  // namespace

extern "C" {

const char *qmm_strerror(int status) {
    switch (status) {
    case QMM_OK: return "ok";
    case QMM_ERR_INVALID_ARG: return "invalid argument (null pointer, bad handle or unknown dtype)";
    case QMM_ERR_UNSUPPORTED: return "dtype not supported by this call";
    case QMM_ERR_SHAPE: return "size out of range, or k not a whole number of blocks";
    case QMM_ERR_ALIGN: return "pointer not 16-byte aligned";
    case QMM_ERR_ARCH: return "device is not sm_103 (GB300)";
    case QMM_ERR_CUDA: return "a CUDA runtime call failed";
    case QMM_ERR_TIMEOUT: return "a device-side bounded wait expired";
    case QMM_ERR_WORKSPACE: return "workspace missing or too small";
    case QMM_ERR_OVERLAP: return "an output buffer overlaps an input buffer";
    default: return "unknown status";
    }
}

int64_t qmm_block_weights(qmm_dtype t) {
    switch (t) {
    case QMM_F32: return 1;
    case QMM_Q4_0: return 32;
    case QMM_Q8_0: return 32;
    case QMM_Q4_K: return 256;
    case QMM_Q6_K: return 256;
    case QMM_NVFP4: return 64;
    case QMM_NVFP4_V2: return 32;
    default: return 0;
    }
}

int64_t qmm_block_bytes(qmm_dtype t) {
    switch (t) {
    case QMM_F32: return 4;
    case QMM_Q4_0: return 18;
    case QMM_Q8_0: return 34;
    case QMM_Q4_K: return 144;
    case QMM_Q6_K: return 210;
    case QMM_NVFP4: return 36;
    case QMM_NVFP4_V2: return 18;
    default: return 0;
    }
}

int64_t qmm_row_bytes(qmm_dtype t, int64_t k) {
    const int64_t qk = qmm_block_weights(t);
    if (qk == 0 || k < 1 || k % qk != 0) return 0;
    return k / qk * qmm_block_bytes(t);
}

size_t qmm_gemm_workspace_bytes(qmm_dtype t, int64_t /*m*/, int64_t k, int64_t n) {
    if (!known_dtype(t) || t == QMM_F32 || t == QMM_NVFP4_V2 || n <= QMM_GEMV_MAX_N || k < 1 || n < 1) return 0;
    const size_t b = static_cast<size_t>(n) * static_cast<size_t>(k) * 2u;
    return (b + 255u) & ~size_t(255);
}

int qmm_create(int device, qmm_handle *out) {
    if (!out) return QMM_ERR_INVALID_ARG;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) return QMM_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return QMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return QMM_ERR_ARCH;
    qmm_ctx *h = static_cast<qmm_ctx *>(calloc(1, sizeof(qmm_ctx)));
    if (!h) return QMM_ERR_CUDA;
    h->magic = kMagic;
    h->device = device;
    h->num_sms = prop.multiProcessorCount;
    h->wait_limit_ns = kDefaultWaitLimitNs;
    const int st = on_device(h, [&]() -> cudaError_t {
        cudaError_t e = cudaMalloc(&h->d_status, sizeof(uint32_t));
        if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(uint32_t));
        if (e == cudaSuccess) e = qmm::gemm_tc_init();
        if (e == cudaSuccess) e = qmm::gemm_fp4_init();
        return e;
    });
    if (st != QMM_OK) {
        if (h->d_status) cudaFree(h->d_status);
        free(h);
        return st;
    }
    *out = h;
    return QMM_OK;
}

int qmm_destroy(qmm_handle h) {
    if (!h) return QMM_OK;
    if (!valid_handle(h)) return QMM_ERR_INVALID_ARG;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(h->device);
    cudaFree(h->d_status);
    if (prev >= 0) cudaSetDevice(prev);
    h->magic = 0;
    free(h);
    return QMM_OK;
}

int qmm_gemv(qmm_handle h, qmm_dtype t, const void *w, const float *x, float *dst, int64_t m, int64_t k, int64_t n,
             void *stream) {
    int st = check_product(h, t, w, x, dst, m, k, n);
    if (st != QMM_OK) return st;
    if (n > QMM_GEMV_MAX_N) return QMM_ERR_SHAPE;
    const int64_t rb = qmm_row_bytes(t, k);
    return on_device(h, [&] {
        return qmm::launch_gemv(t, w, rb, x, dst, m, k, static_cast<int>(n), h->num_sms, h->d_status,
                                h->wait_limit_ns, static_cast<cudaStream_t>(stream));
    });
}

int qmm_gemm(qmm_handle h, qmm_dtype t, const void *w, const float *x, float *dst, int64_t m, int64_t k, int64_t n,
             void *workspace, size_t workspace_bytes, void *stream) {
    int st = check_product(h, t, w, x, dst, m, k, n);
    if (st != QMM_OK) return st;
    if (n <= QMM_GEMV_MAX_N) return qmm_gemv(h, t, w, x, dst, m, k, n, stream);
    if (t == QMM_NVFP4_V2) return QMM_ERR_UNSUPPORTED;  // the tensor-core decode reads 36-byte groups
    if (t == QMM_F32 && k % 4 != 0) return QMM_ERR_SHAPE;  // TMA row pitch must be a multiple of 16 bytes
    const size_t need = qmm_gemm_workspace_bytes(t, m, k, n);
    if (need) {
        if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned16(workspace)) return QMM_ERR_ALIGN;
        if (overlaps(workspace, need, dst, static_cast<size_t>(n * m) * sizeof(float)) ||
            overlaps(workspace, need, x, static_cast<size_t>(n * k) * sizeof(float)) ||
            overlaps(workspace, need, w, static_cast<size_t>(qmm_row_bytes(t, k) * m)))
            return QMM_ERR_OVERLAP;
    }
    qmm::GemmArgs a;
    a.dtype = t;
    a.w = w;
    a.rb = qmm_row_bytes(t, k);
    a.x = x;
    a.dst = dst;
    a.m = m;
    a.k = k;
    a.n = n;
    a.x16 = workspace;
    a.status = h->d_status;
    a.wait_limit_ns = h->wait_limit_ns;
    a.debug_skip_first_b_load = h->debug_skip_first_b_load;
    return on_device(h, [&] { return qmm::launch_gemm_tc(a, h->num_sms, static_cast<cudaStream_t>(stream)); });
}

int qmm_moe_gemv(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales, const float *x, float *y,
                 int64_t in_f, int64_t n_ff, int n_used, int t_tokens, void *stream) {
    if (!valid_handle(h) || !known_dtype(t) || !w_ptrs || !scales || !x || !y) return QMM_ERR_INVALID_ARG;
    if (n_used < 1 || t_tokens < 1 || static_cast<int64_t>(n_used) * t_tokens > 4096) return QMM_ERR_SHAPE;
    if (n_ff < 1 || n_ff > kMaxMN || in_f < 1 || in_f > kMaxK || !k_ok(t, in_f)) return QMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(w_ptrs) & 7u) != 0 || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0 ||
        !aligned16(x) || !aligned16(y))
        return QMM_ERR_ALIGN;
    const int n_pairs = n_used * t_tokens;
    const size_t ybytes = static_cast<size_t>(2) * n_pairs * n_ff * sizeof(float);
    if (overlaps(y, ybytes, x, static_cast<size_t>(t_tokens) * in_f * sizeof(float)) ||
        overlaps(y, ybytes, scales, static_cast<size_t>(2) * n_pairs * sizeof(float)) ||
        overlaps(y, ybytes, w_ptrs, static_cast<size_t>(2) * n_pairs * sizeof(void *)))
        return QMM_ERR_OVERLAP;
    const int64_t rb = qmm_row_bytes(t, in_f);
    return on_device(h, [&] {
        return qmm::launch_moe_gemv(t, w_ptrs, rb, scales, x, y, in_f, n_ff, n_used, n_pairs, t_tokens, h->num_sms,
                                    h->d_status, h->wait_limit_ns, static_cast<cudaStream_t>(stream));
    });
}

size_t qmm_moe_down_workspace_bytes(int64_t gin, int n_used, int t_tokens) {
    if (gin < 1 || n_used <= 1 || t_tokens < 1) return 0;
    const size_t b = static_cast<size_t>(n_used) * static_cast<size_t>(t_tokens) * static_cast<size_t>(gin) * 4u;
    return (b + 255u) & ~size_t(255);
}

int qmm_moe_down(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales, const float *hact,
                 float *y, int64_t n_ff, int64_t gin, int n_used, int t_tokens, void *workspace,
                 size_t workspace_bytes, void *stream) {
    if (!valid_handle(h) || !known_dtype(t) || !w_ptrs || !scales || !hact || !y) return QMM_ERR_INVALID_ARG;
    if (n_used < 1 || t_tokens < 1 || static_cast<int64_t>(n_used) * t_tokens > 4096) return QMM_ERR_SHAPE;
    if (gin < 1 || gin > kMaxMN || n_ff < 1 || n_ff > kMaxK || !k_ok(t, n_ff)) return QMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(w_ptrs) & 7u) != 0 || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0 ||
        !aligned16(hact) || !aligned16(y))
        return QMM_ERR_ALIGN;
    const int n_pairs = n_used * t_tokens;
    const size_t ybytes = static_cast<size_t>(t_tokens) * gin * sizeof(float);
    const size_t hbytes = static_cast<size_t>(n_pairs) * n_ff * sizeof(float);
    const size_t sbytes = static_cast<size_t>(n_pairs) * sizeof(float);
    const size_t pbytes = static_cast<size_t>(n_pairs) * sizeof(void *);
    if (overlaps(y, ybytes, hact, hbytes) || overlaps(y, ybytes, scales, sbytes) || overlaps(y, ybytes, w_ptrs, pbytes))
        return QMM_ERR_OVERLAP;
    const size_t need = qmm_moe_down_workspace_bytes(gin, n_used, t_tokens);
    if (need) {
        if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned16(workspace)) return QMM_ERR_ALIGN;
        if (overlaps(workspace, need, y, ybytes) || overlaps(workspace, need, hact, hbytes) ||
            overlaps(workspace, need, scales, sbytes) || overlaps(workspace, need, w_ptrs, pbytes))
            return QMM_ERR_OVERLAP;
    }
    const int64_t rb = qmm_row_bytes(t, n_ff);
    return on_device(h, [&] {
        return qmm::launch_moe_down(t, w_ptrs, rb, scales, hact, y, static_cast<float *>(workspace), n_ff, gin,
                                    n_used, t_tokens, h->num_sms, h->d_status, h->wait_limit_ns,
                                    static_cast<cudaStream_t>(stream));
    });
}

int qmm_quantize_q8_1(qmm_handle h, const float *x, int8_t *q, float *d, int64_t rows, int64_t k, void *stream) {
    if (!valid_handle(h) || !x || !q || !d) return QMM_ERR_INVALID_ARG;
    if (rows < 1 || rows > kMaxMN || k < 32 || k > kMaxK || k % 32 != 0) return QMM_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(d)) return QMM_ERR_ALIGN;
    const size_t xbytes = static_cast<size_t>(rows * k) * sizeof(float);
    const size_t qbytes = static_cast<size_t>(rows * k), dbytes = static_cast<size_t>(rows * (k / 32)) * sizeof(float);
    if (overlaps(q, qbytes, x, xbytes) || overlaps(d, dbytes, x, xbytes) || overlaps(q, qbytes, d, dbytes))
        return QMM_ERR_OVERLAP;
    return on_device(h, [&] {
        return qmm::launch_quantize_q8_1(x, q, d, rows, k, h->num_sms, static_cast<cudaStream_t>(stream));
    });
}

int qmm_moe_gemv_q8(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales, const int8_t *q,
                    const float *d, float *y, int64_t in_f, int64_t n_ff, int n_used, int t_tokens, void *stream) {
    if (!valid_handle(h) || !known_dtype(t) || !w_ptrs || !scales || !q || !d || !y) return QMM_ERR_INVALID_ARG;
    if (t != QMM_NVFP4 && t != QMM_NVFP4_V2) return QMM_ERR_UNSUPPORTED;
    if (n_used < 1 || t_tokens < 1 || static_cast<int64_t>(n_used) * t_tokens > 4096) return QMM_ERR_SHAPE;
    if (n_ff < 1 || n_ff > kMaxMN || in_f < 64 || in_f > QMM_Q8_MAX_K || in_f % 64 != 0) return QMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(w_ptrs) & 7u) != 0 || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0 ||
        !aligned16(q) || !aligned16(d) || !aligned16(y))
        return QMM_ERR_ALIGN;
    const int n_pairs = n_used * t_tokens;
    const size_t ybytes = static_cast<size_t>(2) * n_pairs * n_ff * sizeof(float);
    if (overlaps(y, ybytes, q, static_cast<size_t>(t_tokens) * in_f) ||
        overlaps(y, ybytes, d, static_cast<size_t>(t_tokens) * (in_f / 32) * sizeof(float)) ||
        overlaps(y, ybytes, scales, static_cast<size_t>(2) * n_pairs * sizeof(float)) ||
        overlaps(y, ybytes, w_ptrs, static_cast<size_t>(2) * n_pairs * sizeof(void *)))
        return QMM_ERR_OVERLAP;
    const int64_t rb = qmm_row_bytes(t, in_f);
    return on_device(h, [&] {
        return qmm::launch_moe_q8(t, w_ptrs, rb, scales, q, d, nullptr, y, in_f, n_ff, 2 * n_pairs, n_pairs, n_used,
                                  h->num_sms, h->d_status, h->wait_limit_ns, static_cast<cudaStream_t>(stream));
    });
}

int qmm_moe_gemv_q8_fused(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales, const float *x,
                          float *y, int64_t in_f, int64_t n_ff, int n_used, int t_tokens, void *stream) {
    if (!valid_handle(h) || !known_dtype(t) || !w_ptrs || !scales || !x || !y) return QMM_ERR_INVALID_ARG;
    if (t != QMM_NVFP4 && t != QMM_NVFP4_V2) return QMM_ERR_UNSUPPORTED;
    if (n_used < 1 || t_tokens < 1 || static_cast<int64_t>(n_used) * t_tokens > 4096) return QMM_ERR_SHAPE;
    if (n_ff < 1 || n_ff > kMaxMN || in_f < 64 || in_f > QMM_Q8_MAX_K || in_f % 64 != 0) return QMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(w_ptrs) & 7u) != 0 || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0 ||
        !aligned16(x) || !aligned16(y))
        return QMM_ERR_ALIGN;
    const int n_pairs = n_used * t_tokens;
    const size_t ybytes = static_cast<size_t>(2) * n_pairs * n_ff * sizeof(float);
    if (overlaps(y, ybytes, x, static_cast<size_t>(t_tokens) * in_f * sizeof(float)) ||
        overlaps(y, ybytes, scales, static_cast<size_t>(2) * n_pairs * sizeof(float)) ||
        overlaps(y, ybytes, w_ptrs, static_cast<size_t>(2) * n_pairs * sizeof(void *)))
        return QMM_ERR_OVERLAP;
    const int64_t rb = qmm_row_bytes(t, in_f);
    return on_device(h, [&] {
        return qmm::launch_moe_q8(t, w_ptrs, rb, scales, nullptr, nullptr, x, y, in_f, n_ff, 2 * n_pairs, n_pairs,
                                  n_used, h->num_sms, h->d_status, h->wait_limit_ns, static_cast<cudaStream_t>(stream));
    });
}

// The down projection on Q8_1 activations: given as (q, d), or as x float32
// quantized inside the kernel (q = d = NULL).
static int moe_down_q8_impl(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales,
                            const int8_t *q, const float *d, const float *x, float *y, int64_t n_ff, int64_t gin,
                            int n_used, int t_tokens, void *workspace, size_t workspace_bytes, void *stream) {
    if (!valid_handle(h) || !known_dtype(t) || !w_ptrs || !scales || !y || (x ? (q || d) : (!q || !d)))
        return QMM_ERR_INVALID_ARG;
    if (t != QMM_NVFP4 && t != QMM_NVFP4_V2) return QMM_ERR_UNSUPPORTED;
    if (n_used < 1 || t_tokens < 1 || static_cast<int64_t>(n_used) * t_tokens > 4096) return QMM_ERR_SHAPE;
    if (gin < 1 || gin > kMaxMN || n_ff < 64 || n_ff > QMM_Q8_MAX_K || n_ff % 64 != 0) return QMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(w_ptrs) & 7u) != 0 || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0 ||
        (x ? !aligned16(x) : (!aligned16(q) || !aligned16(d))) || !aligned16(y))
        return QMM_ERR_ALIGN;
    const int n_pairs = n_used * t_tokens;
    const size_t ybytes = static_cast<size_t>(t_tokens) * gin * sizeof(float);
    const size_t qbytes = x ? 0 : static_cast<size_t>(n_pairs) * n_ff;
    const size_t dbytes = x ? 0 : static_cast<size_t>(n_pairs) * (n_ff / 32) * sizeof(float);
    const size_t xbytes = x ? static_cast<size_t>(n_pairs) * n_ff * sizeof(float) : 0;
    const size_t sbytes = static_cast<size_t>(n_pairs) * sizeof(float);
    const size_t pbytes = static_cast<size_t>(n_pairs) * sizeof(void *);
    if (overlaps(y, ybytes, q, qbytes) || overlaps(y, ybytes, d, dbytes) || overlaps(y, ybytes, x, xbytes) ||
        overlaps(y, ybytes, scales, sbytes) || overlaps(y, ybytes, w_ptrs, pbytes))
        return QMM_ERR_OVERLAP;
    const size_t need = qmm_moe_down_workspace_bytes(gin, n_used, t_tokens);
    if (need) {
        if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned16(workspace)) return QMM_ERR_ALIGN;
        if (overlaps(workspace, need, y, ybytes) || overlaps(workspace, need, q, qbytes) ||
            overlaps(workspace, need, d, dbytes) || overlaps(workspace, need, x, xbytes) ||
            overlaps(workspace, need, scales, sbytes) || overlaps(workspace, need, w_ptrs, pbytes))
            return QMM_ERR_OVERLAP;
    }
    const int64_t rb = qmm_row_bytes(t, n_ff);
    return on_device(h, [&]() -> cudaError_t {
        // the pair products (activation row = pair), then the per-token combine
        float *part = n_used == 1 ? y : static_cast<float *>(workspace);
        cudaError_t e = qmm::launch_moe_q8(t, w_ptrs, rb, scales, q, d, x, part, n_ff, gin, n_pairs, n_pairs, 1,
                                           h->num_sms, h->d_status, h->wait_limit_ns,
                                           static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess || n_used == 1) return e;
        return qmm::launch_moe_combine(part, y, gin, n_used, t_tokens, h->num_sms, static_cast<cudaStream_t>(stream));
    });
}

int qmm_moe_down_q8(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales, const int8_t *q,
                    const float *d, float *y, int64_t n_ff, int64_t gin, int n_used, int t_tokens, void *workspace,
                    size_t workspace_bytes, void *stream) {
    if (!q || !d) return QMM_ERR_INVALID_ARG;
    return moe_down_q8_impl(h, t, w_ptrs, scales, q, d, nullptr, y, n_ff, gin, n_used, t_tokens, workspace,
                            workspace_bytes, stream);
}

int qmm_moe_down_q8_fused(qmm_handle h, qmm_dtype t, const void *const *w_ptrs, const float *scales, const float *x,
                          float *y, int64_t n_ff, int64_t gin, int n_used, int t_tokens, void *workspace,
                          size_t workspace_bytes, void *stream) {
    if (!x) return QMM_ERR_INVALID_ARG;
    return moe_down_q8_impl(h, t, w_ptrs, scales, nullptr, nullptr, x, y, n_ff, gin, n_used, t_tokens, workspace,
                            workspace_bytes, stream);
}

int qmm_quantize_nvfp4(qmm_handle h, const float *x, void *xq, int64_t rows, int64_t k, void *stream) {
    if (!valid_handle(h) || !x || !xq) return QMM_ERR_INVALID_ARG;
    if (rows < 1 || rows > kMaxMN || k < 256 || k > kMaxK || k % 256 != 0) return QMM_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(xq)) return QMM_ERR_ALIGN;
    if (overlaps(xq, static_cast<size_t>(rows * qmm_row_bytes(QMM_NVFP4_V2, k)), x,
                 static_cast<size_t>(rows * k) * sizeof(float)))
        return QMM_ERR_OVERLAP;
    return on_device(h, [&] {
        return qmm::launch_quantize_nvfp4(x, xq, rows, k, h->num_sms, static_cast<cudaStream_t>(stream));
    });
}

int qmm_gemm_fp4(qmm_handle h, const void *w, const void *xq, float *dst, int64_t m, int64_t k, int64_t n,
                 void *stream) {
    if (!valid_handle(h) || !w || !xq || !dst) return QMM_ERR_INVALID_ARG;
    if (m < 1 || n < 1 || m > kMaxMN || n > kMaxMN || k < 256 || k > kMaxK || k % 256 != 0) return QMM_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(xq) || !aligned16(dst)) return QMM_ERR_ALIGN;
    const int64_t rb = qmm_row_bytes(QMM_NVFP4_V2, k);
    const size_t dbytes = static_cast<size_t>(n * m) * sizeof(float);
    if (overlaps(dst, dbytes, w, static_cast<size_t>(rb * m)) || overlaps(dst, dbytes, xq, static_cast<size_t>(rb * n)))
        return QMM_ERR_OVERLAP;
    return on_device(h, [&] {
        return qmm::launch_gemm_fp4(w, xq, dst, m, k, n, h->num_sms, h->d_status, h->wait_limit_ns,
                                    static_cast<cudaStream_t>(stream));
    });
}

int qmm_dequant(qmm_handle h, qmm_dtype t, const void *w, float *out, int64_t m, int64_t k, float tensor_scale,
                void *stream) {
    if (!valid_handle(h) || !known_dtype(t) || !w || !out) return QMM_ERR_INVALID_ARG;
    if (m < 1 || m > kMaxMN || k < 1 || k > kMaxK || !k_ok(t, k)) return QMM_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(out)) return QMM_ERR_ALIGN;
    if (overlaps(out, static_cast<size_t>(m * k) * sizeof(float), w, static_cast<size_t>(qmm_row_bytes(t, k) * m)))
        return QMM_ERR_OVERLAP;
    const int64_t rb = qmm_row_bytes(t, k);
    return on_device(h, [&] {
        return qmm::launch_dequant(t, w, out, m, k, rb, tensor_scale, h->num_sms, static_cast<cudaStream_t>(stream));
    });
}

int qmm_nvfp4_repack_v2(qmm_handle h, const void *v1, void *v2, int64_t m, int64_t k, void *stream) {
    if (!valid_handle(h) || !v1 || !v2) return QMM_ERR_INVALID_ARG;
    if (m < 1 || m > kMaxMN || k < 64 || k > kMaxK || k % 64 != 0) return QMM_ERR_SHAPE;
    if (!aligned16(v1) || !aligned16(v2)) return QMM_ERR_ALIGN;
    const size_t bytes = static_cast<size_t>(qmm_row_bytes(QMM_NVFP4, k) * m);
    if (overlaps(v1, bytes, v2, bytes)) return QMM_ERR_OVERLAP;
    return on_device(h, [&] {
        return qmm::launch_nvfp4_repack_v2(static_cast<const uint8_t *>(v1), static_cast<uint8_t *>(v2), m, k,
                                           h->num_sms, static_cast<cudaStream_t>(stream));
    });
}

int qmm_sync_status(qmm_handle h, void *stream) {
    if (!valid_handle(h)) return QMM_ERR_INVALID_ARG;
    uint32_t bits = 0;
    const int st = on_device(h, [&]() -> cudaError_t {
        cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) e = cudaMemcpy(&bits, h->d_status, sizeof(bits), cudaMemcpyDeviceToHost);
        if (e == cudaSuccess && bits) e = cudaMemset(h->d_status, 0, sizeof(uint32_t));
        return e;
    });
    if (st != QMM_OK) return st;
    if (bits & 1u) return QMM_ERR_TIMEOUT;
    if (bits & 2u) return QMM_ERR_ALIGN;
    return QMM_OK;
}

// ---- test hooks (include/qmm_testing.h) ----

int qmm_testing_set_wait_limit_ns(qmm_handle h, uint64_t limit_ns) {
    if (!valid_handle(h) || limit_ns == 0) return QMM_ERR_INVALID_ARG;
    h->wait_limit_ns = limit_ns;
    return QMM_OK;
}

int qmm_testing_skip_first_stage_load(qmm_handle h, int enable) {
    if (!valid_handle(h)) return QMM_ERR_INVALID_ARG;
    h->debug_skip_first_b_load = enable ? 1 : 0;
    return QMM_OK;
}

}  // extern "C"
