// dequant.cu -- standalone packed -> float32 dequant (the dequantize-to-FP32
// step of the v1 prefill path in aprender-serve 0.70.2 cublas_prefill/mod.rs,
// module doc).
//
// One thread decodes 8 consecutive weights into a shared buffer; each CTA's
// chunk of 128 groups leaves in one bulk store; the grid strides over the
// chunks.  The file also holds the
// repack of NVFP4 rows into the V2 layout (a byte permutation).  Bit-exact: every value is
// the format's value rounded once to float32 (decode.cuh).
#include "kernels.h"
#include "decode.cuh"
#include "l2hint.cuh"

namespace qmm {

// 1-D bulk store shared -> global (the TMA engine), tracked by the issuing
// thread's bulk groups; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void dq_bulk_store_nocommit(void *gdst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(gdst)),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void dq_bulk_store(void *gdst, const void *smem_src, uint32_t bytes) {
    dq_bulk_store_nocommit(gdst, smem_src, bytes);
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Chunks of 128 consecutive 8-weight groups (4 KB of output, contiguous:
// group g's values are out[8g .. 8g+7]) for CTAs of 128 threads: thread t
// decodes group t of the chunk into a shared buffer, and one bulk store
// writes the chunk, so the fp32 stream leaves through the TMA engine instead
// of 256 per-thread stores.  Two buffers: a chunk's buffer is reused two
// chunks later, once its store has read it.  (Chunks of 256 groups for
// 256-thread CTAs ran 2-3 % slower.)
template <typename Idx, typename Decode>
__device__ __forceinline__ void dequant_chunks(float *__restrict__ out, Idx total, Decode decode) {
    constexpr int T = 128;
    __shared__ __align__(128) float4 buf[2][2 * T];
    const Idx nchunks = (total + T - 1) / T;
    int b = 0;
    for (Idx c = blockIdx.x; c < nchunks; c += gridDim.x, b ^= 1) {
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const Idx g = c * T + threadIdx.x;
        if (g < total) {
            float v[8];
            decode(g, v);
            buf[b][2 * threadIdx.x] = make_float4(v[0], v[1], v[2], v[3]);
            buf[b][2 * threadIdx.x + 1] = make_float4(v[4], v[5], v[6], v[7]);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            const Idx n = total - c * T < T ? total - c * T : T;
            dq_bulk_store(out + c * T * 8, &buf[b][0], static_cast<uint32_t>(n) * 32u);
        }
    }
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <int F, typename Idx>
__global__ void __launch_bounds__(128) dequant_kernel(const uint8_t *__restrict__ w, float *__restrict__ out,
                                                      Idx m, Idx k, Idx rb, float ts) {
    constexpr int QK = Fmt<F>::QK, BB = Fmt<F>::BB;
    // an equal slice of the packed weights into L2 per CTA, before waiting
    // for the kernel in front (a cache hint; the loads after the wait hit L2)
    if (threadIdx.x == 0) {
        const uint64_t wb = static_cast<uint64_t>(m) * static_cast<uint64_t>(rb);
        const uint64_t chunk = (wb + gridDim.x - 1) / gridDim.x;
        const uint64_t b0 = static_cast<uint64_t>(blockIdx.x) * chunk;
        const uint64_t b1 = b0 + chunk < wb ? b0 + chunk : wb;
        if (b0 < b1)
            prefetch_l2_range(reinterpret_cast<uintptr_t>(w) + b0, reinterpret_cast<uintptr_t>(w) + b1);
    }
    griddep_wait();
    griddep_launch();
    const Idx gpr = k / 8;  // groups per row
    dequant_chunks(out, m * gpr, [&](Idx g, float (&v)[8]) {
        const Idx r = g / gpr;
        const Idx e0 = (g - r * gpr) * 8;
        Dec8<F, LdG>::run(w + r * rb + (e0 / QK) * BB, static_cast<int>(e0 % QK), ts, v);
    });
}

// f32 weights: the decoded value is the weight itself.
__global__ void __launch_bounds__(256) copy_f32_kernel(const float *__restrict__ w, float *__restrict__ out,
                                                       int64_t n) {
    griddep_wait();
    griddep_launch();
    const int64_t n4 = n / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
        reinterpret_cast<float4 *>(out)[i] = __ldg(reinterpret_cast<const float4 *>(w) + i);
    for (int64_t i = 4 * n4 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = __ldg(w + i);
}

// NVFP4 V2 rows (k/2 code bytes, then k/16 E4M3 scale bytes; k % 64 == 0,
// so every row starts on a 4-byte boundary): one thread decodes 8
// consecutive weights from one code word and one scale byte, each value
// (e2m1 * e4m3, exact) times ts rounded once, as for the 36-byte groups.
__global__ void __launch_bounds__(128) dequant_nvfp4_v2_kernel(const uint8_t *__restrict__ w,
                                                               float *__restrict__ out, int64_t m, int64_t k,
                                                               float ts) {
    const int64_t rb = k / 32 * 18;
    if (threadIdx.x == 0) {
        const uint64_t wb = static_cast<uint64_t>(m) * static_cast<uint64_t>(rb);
        const uint64_t chunk = (wb + gridDim.x - 1) / gridDim.x;
        const uint64_t b0 = static_cast<uint64_t>(blockIdx.x) * chunk;
        const uint64_t b1 = b0 + chunk < wb ? b0 + chunk : wb;
        if (b0 < b1)
            prefetch_l2_range(reinterpret_cast<uintptr_t>(w) + b0, reinterpret_cast<uintptr_t>(w) + b1);
    }
    griddep_wait();
    griddep_launch();
    const int64_t gpr = k / 8;
    dequant_chunks(out, m * gpr, [&](int64_t g, float (&v)[8]) {
        const int64_t r = g / gpr;
        const int64_t e0 = (g - r * gpr) * 8;
        const uint8_t *row = w + r * rb;
        const uint32_t codes = __ldg(reinterpret_cast<const unsigned int *>(row + e0 / 2));
        const float s = e4m3_to_f32(__ldg(row + k / 2 + e0 / 16));
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(__fmul_rn(e2m1_to_f32((codes >> (4 * j)) & 15u), s), ts);
    });
}

// NVFP4 36-byte groups -> V2 rows: one thread moves one group (nine 4-byte
// words; rows of k/64*36 bytes keep every group 4-byte aligned), its 32 code
// bytes to 32g of the row and its 4 scale bytes to k/2 + 4g.
__global__ void __launch_bounds__(256) nvfp4_repack_v2_kernel(const uint8_t *__restrict__ v1,
                                                              uint8_t *__restrict__ v2, int64_t m, int64_t k) {
    griddep_wait();
    griddep_launch();
    const int64_t gpr = k / 64, rb = gpr * 36, total = m * gpr;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = g / gpr, q = g - r * gpr;
        const unsigned int *src = reinterpret_cast<const unsigned int *>(v1 + r * rb + q * 36);
        unsigned int *codes = reinterpret_cast<unsigned int *>(v2 + r * rb + q * 32);
        unsigned int *scales = reinterpret_cast<unsigned int *>(v2 + r * rb + k / 2 + q * 4);
        *scales = __ldg(src);
#pragma unroll
        for (int j = 0; j < 8; ++j) codes[j] = __ldg(src + 1 + j);
    }
}

// The same repack for k % 256 == 0 (rows of a multiple of 16 bytes, groups
// per row a multiple of 4): chunks of 256 consecutive groups, thread t
// loading group t and placing its code words and scale word into shared
// buffers laid out as the V2 row segments; then thread j writes the chunk's
// part of row j of the chunk with two bulk stores (codes, scales), all
// 16-byte aligned because every segment starts and ends on a group index
// that is a multiple of 4.  Two buffer pairs; a pair is reused once the
// stores that read it (each by the thread that issued them) are done.
__global__ void __launch_bounds__(256) nvfp4_repack_v2_chunks_kernel(const uint8_t *__restrict__ v1,
                                                                     uint8_t *__restrict__ v2, int64_t m,
                                                                     int64_t k) {
    __shared__ __align__(128) uint4 cbuf[2][2 * 256];  // code words, 32 bytes per group
    __shared__ __align__(128) unsigned int sbuf[2][256];  // scale words
    griddep_wait();
    griddep_launch();
    const int64_t gpr = k / 64, rb = gpr * 36, total = m * gpr;
    const int64_t nchunks = (total + 255) / 256;
    int b = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, b ^= 1) {
        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const int64_t g0 = c * 256, g1 = g0 + 256 < total ? g0 + 256 : total;
        const int64_t g = g0 + threadIdx.x;
        if (g < g1) {  // rows are contiguous: group g starts at 36 g
            const unsigned int *src = reinterpret_cast<const unsigned int *>(v1 + g * 36);
            sbuf[b][threadIdx.x] = __ldg(src);
            cbuf[b][2 * threadIdx.x] = make_uint4(__ldg(src + 1), __ldg(src + 2), __ldg(src + 3), __ldg(src + 4));
            cbuf[b][2 * threadIdx.x + 1] = make_uint4(__ldg(src + 5), __ldg(src + 6), __ldg(src + 7), __ldg(src + 8));
        }
        fence_proxy_async_smem();
        __syncthreads();
        const int64_t r = g0 / gpr + threadIdx.x;  // this thread's row of the chunk
        if (r * gpr < g1) {
            const int64_t qlo = r * gpr < g0 ? g0 - r * gpr : 0;
            const int64_t qhi = (r + 1) * gpr < g1 ? gpr : g1 - r * gpr;
            const int64_t o = r * gpr + qlo - g0;  // the segment's first group within the chunk
            uint8_t *row = v2 + r * rb;
            dq_bulk_store_nocommit(row + qlo * 32, &cbuf[b][2 * o], static_cast<uint32_t>((qhi - qlo) * 32));
            dq_bulk_store_nocommit(row + k / 2 + qlo * 4, &sbuf[b][o], static_cast<uint32_t>((qhi - qlo) * 4));
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

cudaError_t launch_nvfp4_repack_v2(const uint8_t *v1, uint8_t *v2, int64_t m, int64_t k, int num_sms,
                                   cudaStream_t st) {
    const int64_t total = m * (k / 64);
    const int64_t want = (total + 255) / 256;
    const int grid = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
    if (k % 256 == 0 && (reinterpret_cast<uintptr_t>(v2) & 15u) == 0)
        return launch_pdl(nvfp4_repack_v2_chunks_kernel, dim3(grid), dim3(256), 0, st, dim3(1, 1, 1), v1, v2, m, k);
    return launch_pdl(nvfp4_repack_v2_kernel, dim3(grid), dim3(256), 0, st, dim3(1, 1, 1), v1, v2, m, k);
}

template <int F>
static cudaError_t launch_dequant_t(const void *w, float *out, int64_t m, int64_t k, int64_t rb, float ts,
                                    int num_sms, cudaStream_t st) {
    const int64_t total = m * (k / 8);
    const int64_t want = (total + 127) / 128;
    const int grid = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
    if (total < (1LL << 31) && m * k < (1LL << 31))
        return launch_pdl(dequant_kernel<F, uint32_t>, dim3(grid), dim3(128), 0, st, dim3(1, 1, 1), static_cast<const uint8_t *>(w),
                          out, static_cast<uint32_t>(m), static_cast<uint32_t>(k), static_cast<uint32_t>(rb), ts);
    return launch_pdl(dequant_kernel<F, int64_t>, dim3(grid), dim3(128), 0, st, dim3(1, 1, 1), static_cast<const uint8_t *>(w), out,
                      m, k, rb, ts);
}

cudaError_t launch_dequant(int dtype, const void *w, float *out, int64_t m, int64_t k, int64_t rb, float ts,
                           int num_sms, cudaStream_t st) {
    switch (dtype) {
    case QMM_F32: {
        const int64_t n = m * k;
        const int64_t want = (n / 4 + 255) / 256 + 1;
        const int grid = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
        return launch_pdl(copy_f32_kernel, dim3(grid), dim3(256), 0, st, dim3(1, 1, 1), static_cast<const float *>(w), out, n);
    }
    case QMM_Q4_0: return launch_dequant_t<QMM_Q4_0>(w, out, m, k, rb, ts, num_sms, st);
    case QMM_Q8_0: return launch_dequant_t<QMM_Q8_0>(w, out, m, k, rb, ts, num_sms, st);
    case QMM_Q4_K: return launch_dequant_t<QMM_Q4_K>(w, out, m, k, rb, ts, num_sms, st);
    case QMM_Q6_K: return launch_dequant_t<QMM_Q6_K>(w, out, m, k, rb, ts, num_sms, st);
    case QMM_NVFP4: return launch_dequant_t<QMM_NVFP4>(w, out, m, k, rb, ts, num_sms, st);
    case QMM_NVFP4_V2: {
        const int64_t want = (m * (k / 8) + 127) / 128;
        const int grid = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
        return launch_pdl(dequant_nvfp4_v2_kernel, dim3(grid), dim3(128), 0, st, dim3(1, 1, 1),
                          static_cast<const uint8_t *>(w), out, m, k, ts);
    }
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
