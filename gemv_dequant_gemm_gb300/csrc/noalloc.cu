// noalloc.cu -- qmm_gemm_noalloc: qmm_gemm without any device allocation, for
// callers that cannot call cudaMalloc (see include/qmm.h), and
// qmm_gemm_noalloc_status, which reads the device status those calls latch.
// The tensor-core kernel's scratch (the f16 copy of X and a status word)
// lives in one file-scope static device array; the existing launchers do the
// work.
#include <mutex>

#include "../../include/qmm.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratch = QMM_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;  // status word, then the f16 copy of X at a 256-byte offset
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxMN = int64_t(1) << 24;
constexpr int64_t kMaxK = int64_t(1) << 20;

// In host code this name is only a host-side stand-in: the device address
// comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratch];

struct DeviceSetup {
    bool ready;  // set only once every step below has succeeded
    int num_sms;
    unsigned char *scratch;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// Set-up of the current device (with that device current): architecture check,
// kernel attributes, and the device address of the static scratch array.  A
// failure leaves the device not set up, so a later call tries again.  (The
// array itself is zero when its module is placed on the device, so the status
// word starts cleared.)
int setup_current_device(int dev, DeviceSetup **out) {
    if (dev < 0 || dev >= kMaxDevices) return QMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        unsigned char *p = nullptr;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QMM_ERR_CUDA;
        if (major != 10 || minor != 3) return QMM_ERR_ARCH;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return QMM_ERR_CUDA;
        if (qmm::gemm_tc_init() != cudaSuccess) return QMM_ERR_CUDA;
        s.num_sms = sms;
        s.scratch = p;
        s.ready = true;
    }
    *out = &s;
    return QMM_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

}  // namespace

extern "C" int qmm_gemm_noalloc(qmm_dtype t, const void *w, const float *x, float *dst, int64_t m, int64_t k,
                                int64_t n, void *stream) {
    if (!w || !x || !dst || t < QMM_F32 || t > QMM_NVFP4_V2) return QMM_ERR_INVALID_ARG;
    if (m < 1 || n < 1 || m > kMaxMN || n > kMaxMN || k < 1 || k > kMaxK) return QMM_ERR_SHAPE;
    const int64_t rb = qmm_row_bytes(t, k);
    if (rb == 0 || (t == QMM_NVFP4_V2 && k % 64 != 0)) return QMM_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(x) || !aligned16(dst)) return QMM_ERR_ALIGN;
    const size_t dbytes = static_cast<size_t>(n * m) * sizeof(float);
    if (overlaps(dst, dbytes, w, static_cast<size_t>(rb * m)) ||
        overlaps(dst, dbytes, x, static_cast<size_t>(n * k) * sizeof(float)))
        return QMM_ERR_OVERLAP;
    const bool tensor_core = n > QMM_GEMV_MAX_N;
    if (tensor_core && t == QMM_NVFP4_V2) return QMM_ERR_UNSUPPORTED;  // the tensor-core decode reads 36-byte groups
    if (tensor_core && t == QMM_F32 && k % 4 != 0) return QMM_ERR_SHAPE;
    const size_t need = tensor_core ? qmm_gemm_workspace_bytes(t, m, k, n) : 0;
    if (need > kScratch - kStatusBytes) return QMM_ERR_WORKSPACE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
    DeviceSetup *s = nullptr;
    const int st = setup_current_device(dev, &s);
    if (st != QMM_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    // device-side timeouts are OR-ed into the status word until
    // qmm_gemm_noalloc_status reads and clears it
    uint32_t *status = reinterpret_cast<uint32_t *>(s->scratch);
    cudaError_t e;
    if (!tensor_core) {
        e = qmm::launch_gemv(t, w, rb, x, dst, m, k, static_cast<int>(n), s->num_sms, status, 2000000000ull, cs);
    } else {
        qmm::GemmArgs a;
        a.dtype = t;
        a.w = w;
        a.rb = rb;
        a.x = x;
        a.dst = dst;
        a.m = m;
        a.k = k;
        a.n = n;
        a.x16 = s->scratch + kStatusBytes;
        a.status = status;
        a.wait_limit_ns = 2000000000ull;
        a.debug_skip_first_b_load = 0;
        e = qmm::launch_gemm_tc(a, s->num_sms, cs);
    }
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

extern "C" int qmm_gemm_noalloc_status(void *stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
    DeviceSetup *s = nullptr;
    const int st = setup_current_device(dev, &s);
    if (st != QMM_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;  // host stack: no allocation on either side
    if (cudaStreamSynchronize(cs) != cudaSuccess) return QMM_ERR_CUDA;
    if (cudaMemcpy(&bits, s->scratch, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) return QMM_ERR_CUDA;
    if (bits != 0) {
        if (cudaMemsetAsync(s->scratch, 0, sizeof(uint32_t), cs) != cudaSuccess ||
            cudaStreamSynchronize(cs) != cudaSuccess)
            return QMM_ERR_CUDA;
    }
    if (bits & qmm::kDevTimeout) return QMM_ERR_TIMEOUT;
    if (bits & qmm::kDevBadPtr) return QMM_ERR_ALIGN;
    return QMM_OK;
}
