// gemm_tc.cu -- the prefill GEMM dst[n][m] = sum_k W[m][k] X[n][k] on the
// 5th-generation tensor cores (tcgen05), for n > QMM_GEMV_MAX_N.
//
// The product is the one of cera 0.4.0 examples/wgpu_gemm_bench.rs (struct
// Shape: dst[n, m] = src0[m, k] * src1[n, k]; its mul_mat_reg_tile kernel
// decodes src0 blocks into shared memory with per-format loaders).  Here:
//
//   * X (f32) is rounded once to f16 into the caller's workspace by
//     x_to_f16_kernel (round to nearest even, like the cvt.rn.f16.f32
//     converter of aprender-serve cublas_prefill/mod.rs, F32_TO_F16_PTX), and
//     each CTA streams its [BN x 64] f16 tiles with 2-D TMA in the 128-byte
//     swizzled K-major layout the MMA reads.
//   * Packed W is never written back to HBM in decoded form: eight decode
//     warps read each CTA's [BM x 64] weight slice, decode it to f16
//     (decode32_h) and store it straight into the same swizzled layout.
//   * One thread issues tcgen05.mma.kind::f16 (M=128, N=256, K=16; four per
//     64-wide k stage) with fp32 accumulators in tensor memory (256 columns).
//     f32 weights skip the decode: TMA loads W and X as f32 and the MMA runs
//     kind::tf32 (K=8, four per 32-wide stage).
//   * A 4-stage mbarrier ring couples the roles; tcgen05.commit releases a
//     stage when the MMAs that read it are done.
//   * The decode warps then read the accumulator out of TMEM (tcgen05.ld,
//     32 lanes x 32 columns at a time) and store dst[n][m] with m contiguous,
//     so every store instruction writes 128 contiguous bytes.
//
// Every wait is bounded by a wall-clock limit; a wait that runs out latches a
// status bit, the CTA stops issuing work, waits for its own copies and MMAs
// in flight, frees its tensor memory and returns.
#include <cudaTypedefs.h>
#include <string.h>

#include "decode.cuh"
#include "kernels.h"

namespace qmm {

namespace gemm {
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int ROWB = 128;                 // bytes of one operand row in one stage
constexpr int A_STAGE = BM * ROWB;        // 16 KB
constexpr int B_STAGE = BN * ROWB;        // 32 KB
constexpr int NUM_DECODE_WARPS = 8;
constexpr int THREADS = 64 + 32 * NUM_DECODE_WARPS;
constexpr uint32_t TMEM_COLS = 256;

struct Ctl {
    uint64_t full_a[STAGES];  // decode warps finished writing the A stage
    uint64_t full_b[STAGES];  // TMA bytes of the stage landed
    uint64_t empty[STAGES];   // the MMAs reading the stage completed
    uint64_t accum;           // every MMA of the tile completed
    uint32_t tmem_base;
    int abort;
};

constexpr size_t SMEM_BYTES = 1024 + STAGES * (A_STAGE + B_STAGE) + sizeof(Ctl);
}  // namespace gemm

// The same wait with no early exit on abort: used where the thing waited for
// is already in flight (a copy or an MMA) and must land before the CTA ends.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, uint32_t *status, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

template <int F>
__global__ void __launch_bounds__(gemm::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_a,
                   const uint8_t *__restrict__ w, int64_t rb, float *__restrict__ dst, int M, int N, int K,
                   uint32_t *status, uint64_t limit_ns, int debug_skip) {
    using namespace gemm;
    constexpr bool kTF32 = (F == QMM_F32);
    constexpr int KPS = kTF32 ? 32 : 64;  // k elements per stage (128 bytes per row)
    constexpr uint32_t IDESC = mma_idesc(kTF32 ? 2u : 0u, BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = base;
    uint8_t *sB = base + STAGES * A_STAGE;
    Ctl *ctl = reinterpret_cast<Ctl *>(sB + STAGES * B_STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int KT = (K + KPS - 1) / KPS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full_a[s], NUM_DECODE_WARPS);
            mbar_init(&ctl->full_b[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->accum, 1);
        ctl->abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmap_b);
        if (kTF32) prefetch_tensormap(&tmap_a);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int last_kt[STAGES];
            for (int s = 0; s < STAGES; ++s) last_kt[s] = -1;
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                const uint32_t ph = (kt / STAGES) & 1;
                if (!mbar_wait_bounded(&ctl->empty[s], ph ^ 1, abort, status, limit_ns)) break;
                if (debug_skip && kt == 0) continue;  // test hook: stage 0 never fills
                if constexpr (kTF32) {
                    mbar_arrive_expect_tx(&ctl->full_b[s], A_STAGE + B_STAGE);
                    tma_load_2d(sA + s * A_STAGE, &tmap_a, kt * KPS, m0, &ctl->full_b[s]);
                    tma_load_2d(sB + s * B_STAGE, &tmap_b, kt * KPS, n0, &ctl->full_b[s]);
                } else {
                    mbar_arrive_expect_tx(&ctl->full_b[s], B_STAGE);
                    tma_load_2d(sB + s * B_STAGE, &tmap_b, kt * KPS, n0, &ctl->full_b[s]);
                }
                last_kt[s] = kt;
            }
            if (*abort) {
                // let every copy still in flight land before the CTA ends
                for (int s = 0; s < STAGES; ++s)
                    if (last_kt[s] >= 0) mbar_wait_drain(&ctl->full_b[s], (last_kt[s] / STAGES) & 1, status, limit_ns);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                const uint32_t ph = (kt / STAGES) & 1;
                if (!mbar_wait_bounded(&ctl->full_b[s], ph, abort, status, limit_ns)) break;
                if (!kTF32 && !mbar_wait_bounded(&ctl->full_a[s], ph, abort, status, limit_ns)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + s * A_STAGE);
                const uint32_t b_addr = smem_u32(sB + s * B_STAGE);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sw128_desc(a_addr + 32 * kk);
                    const uint64_t bd = sw128_desc(b_addr + 32 * kk);
                    if constexpr (kTF32)
                        mma_tf32(tmem, ad, bd, IDESC, (kt | kk) != 0);
                    else
                        mma_f16(tmem, ad, bd, IDESC, (kt | kk) != 0);
                }
                mma_commit(&ctl->empty[s]);
            }
            // arrives once every MMA issued above has completed
            mma_commit(&ctl->accum);
        }
        __syncwarp();
    } else {
        // ---------------- decode warps, then epilogue ----------------
        const int dt = threadIdx.x - 64;
        if constexpr (!kTF32) {
            const int row = dt & (BM - 1);
            const int half = dt >> 7;  // which 32 of the stage's 64 k
            const int gm = m0 + row;
            const uint8_t *wrow = w + static_cast<int64_t>(gm < M ? gm : 0) * rb;
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                const uint32_t ph = (kt / STAGES) & 1;
                // every lane waits; the vote keeps the exit warp-uniform
                const bool ok = mbar_wait_bounded(&ctl->empty[s], ph ^ 1, abort, status, limit_ns);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                const int64_t e0 = static_cast<int64_t>(kt) * 64 + half * 32;
                uint32_t o[16];
                if (gm < M && e0 < K) {
                    decode32_h<F>(wrow, e0, o);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = 0u;
                }
                uint8_t *rowp = sA + s * A_STAGE + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = half * 4 + j;
                    *reinterpret_cast<uint4 *>(rowp + ((c ^ (row & 7)) << 4)) =
                        make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->full_a[s]);
            }
        }
        // epilogue: wait for the accumulator even after an abort (MMAs may be in flight)
        const bool drained = mbar_wait_drain(&ctl->accum, 0, status, limit_ns);
        // tcgen05.ld is warp-collective: decide for the whole warp
        if (__all_sync(0xFFFFFFFFu, drained && !*abort)) {
            tc_fence_after();
            const int q = warp & 3;
            const int colbase = (warp >= 6) ? BN / 2 : 0;
            const int gm = m0 + 32 * q + lane;
#pragma unroll 1
            for (int c = 0; c < BN / 2 / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + colbase + 32 * c, v);
                tmem_ld_wait();
                const int gn0 = n0 + colbase + 32 * c;
                if (gm < M) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (gn0 + j < N) dst[static_cast<int64_t>(gn0 + j) * M + gm] = __uint_as_float(v[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// X [n][k] f32 -> [n][k] f16, round to nearest even; k % 8 == 0.
__global__ void __launch_bounds__(256) x_to_f16_kernel(const float *__restrict__ x, __half *__restrict__ x16,
                                                       int64_t total8) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total8; i += stride) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(x) + 2 * i);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(x) + 2 * i + 1);
        const __half2 h0 = __floats2half2_rn(a.x, a.y), h1 = __floats2half2_rn(a.z, a.w);
        const __half2 h2 = __floats2half2_rn(b.x, b.y), h3 = __floats2half2_rn(b.z, b.w);
        reinterpret_cast<uint4 *>(x16)[i] = make_uint4(h2_bits(h0), h2_bits(h1), h2_bits(h2), h2_bits(h3));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D tiled map over a row-major [rows][cols] matrix, box [box_rows][box_cols],
// 128-byte swizzle (box_cols * elem == 128), zero fill outside the matrix.
static bool make_map(CUtensorMap *map, const void *base, CUtensorMapDataType dt, int elem, int64_t rows, int64_t cols,
                     int box_rows, int box_cols) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int F>
static cudaError_t launch_gemm_t(const GemmArgs &a, cudaStream_t st) {
    using namespace gemm;
    CUtensorMap map_b, map_a;
    memset(&map_a, 0, sizeof(map_a));
    if (F == QMM_F32) {
        if (!make_map(&map_b, a.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.n, a.k, BN, 32)) return cudaErrorInvalidValue;
        if (!make_map(&map_a, a.w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.m, a.k, BM, 32)) return cudaErrorInvalidValue;
    } else {
        const int64_t total8 = a.n * a.k / 8;
        const int64_t want = (total8 + 255) / 256;
        const int grid = static_cast<int>(want < 1184 ? want : 1184);
        x_to_f16_kernel<<<grid, 256, 0, st>>>(a.x, static_cast<__half *>(a.x16), total8);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (!make_map(&map_b, a.x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.n, a.k, BN, 64)) return cudaErrorInvalidValue;
        map_a = map_b;  // unused by the packed-format kernels
    }
    const dim3 grid(static_cast<unsigned>((a.m + BM - 1) / BM), static_cast<unsigned>((a.n + BN - 1) / BN));
    gemm_tc_kernel<F><<<grid, THREADS, SMEM_BYTES, st>>>(map_b, map_a, static_cast<const uint8_t *>(a.w), a.rb, a.dst,
                                                         static_cast<int>(a.m), static_cast<int>(a.n),
                                                         static_cast<int>(a.k), a.status, a.wait_limit_ns,
                                                         a.debug_skip_first_b_load);
    return cudaGetLastError();
}

// Opt every instance into the large dynamic shared-memory carve-out; called
// once per device (with that device current) when a handle is created.
cudaError_t gemm_tc_init() {
    const int bytes = static_cast<int>(gemm::SMEM_BYTES);
    cudaError_t e = cudaSuccess;
    auto set = [&](const void *fn) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    };
    set(reinterpret_cast<const void *>(gemm_tc_kernel<QMM_F32>));
    set(reinterpret_cast<const void *>(gemm_tc_kernel<QMM_Q4_0>));
    set(reinterpret_cast<const void *>(gemm_tc_kernel<QMM_Q8_0>));
    set(reinterpret_cast<const void *>(gemm_tc_kernel<QMM_Q4_K>));
    set(reinterpret_cast<const void *>(gemm_tc_kernel<QMM_Q6_K>));
    set(reinterpret_cast<const void *>(gemm_tc_kernel<QMM_NVFP4>));
    return e;
}

cudaError_t launch_gemm_tc(const GemmArgs &a, int /*num_sms*/, cudaStream_t st) {
    switch (a.dtype) {
    case QMM_F32: return launch_gemm_t<QMM_F32>(a, st);
    case QMM_Q4_0: return launch_gemm_t<QMM_Q4_0>(a, st);
    case QMM_Q8_0: return launch_gemm_t<QMM_Q8_0>(a, st);
    case QMM_Q4_K: return launch_gemm_t<QMM_Q4_K>(a, st);
    case QMM_Q6_K: return launch_gemm_t<QMM_Q6_K>(a, st);
    case QMM_NVFP4: return launch_gemm_t<QMM_NVFP4>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
