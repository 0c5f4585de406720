// gemm_fp4.cu -- the prefill product on the block-scaled FP4 tensor cores:
// dst[n][m] = sum_k W[m][k] * Xq[n][k] with both W and the activation Xq in
// NVFP4 (E2M1 values, one E4M3 scale per 16 along k), stored as V2 rows
// (k/2 code bytes, then k/16 scale bytes).
//
// memra-engine 0.128.0 moe_rows_ceiling_bench.rs keeps its weights in NVFP4
// groups and, in its V2 arms, as rows whose scales form one contiguous
// stream; aprender-serve 0.70.2 cublas_prefill/mod.rs routes its prefill to a
// lower-precision tensor-core GEMM with a quantized activation scratch.  Here
// the tcgen05 MMA of kind mxf4nvf4 reads the packed codes and applies the
// E4M3 scales itself (scale_vec::4X: four scales per row per K = 64 MMA), so
// nothing is decoded in software: each product of two E2M1 values is exact,
// a 16-term block sum is exact, it is scaled by the two E4M3 scales and
// accumulated in fp32 in tensor memory.
//
// CTA = one 128 (m) x 128 (n) output tile, k in 256-wide stages (split
// over a cluster of up to 8 CTAs when the tiles alone do not cover the SMs):
//   warp 0      TMA producer: per stage the W and X code tiles (128 rows x
//               128 bytes each, 128-byte swizzle: the K-major operand layout)
//               and the W and X scale tiles (128 rows x 16 bytes);
//   warp 1      TMEM allocation and the MMA-issuing thread: four K = 64
//               MMAs per stage, A = W codes, B = X codes, scales from TMEM;
//   warps 2-5   scale movers: the stage's scale tiles go to tensor memory in
//               the MMA's scale layout (rows 32i + j in column i of lane j,
//               the same in every lane quarter, four columns per MMA), one
//               tcgen05.st of 16 columns per operand and warp; then the
//               epilogue: tcgen05.ld of the fp32 accumulator into shared
//               memory as [n][m], a TMA store per 32 columns (split-K: a
//               fixed-order sum of the cluster's partial tiles through
//               distributed shared memory, no atomics).
// Every wait is bounded; a wait that runs out latches the timeout bit and
// the CTA stops issuing work, waits for its copies and MMAs in flight, frees
// its tensor memory and returns without storing.
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

#include "decode.cuh"
#include "kernels.h"

namespace qmm {

namespace f4 {
constexpr int BM = 128, BN = 128;
constexpr int KS = 256;                  // k per stage
constexpr int CODE_TILE = 128 * 128;     // bytes: 128 rows x 128 code bytes (256 values)
constexpr int SCALE_TILE = 128 * 16;     // bytes: 128 rows x 16 scale bytes
constexpr int STAGE = 2 * CODE_TILE + 2 * SCALE_TILE;
constexpr int STAGES = 5;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;           // 128 accumulator columns, then the scale columns
// Scale columns of stage slot s: W at SF_COL0 + 32s, X at SF_COL0 + 32s + 16;
// MMA kk of the stage reads four columns from + 4kk.  In those four columns,
// lane j (of every lane quarter) holds in column i the four scales of row
// 32i + j for the MMA's four 16-wide k blocks, byte b for block b.
constexpr int SF_COL0 = 128;
constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE + 256;

struct Ctl {
    uint64_t full[STAGES], sf_full[STAGES], empty[STAGES];
    uint64_t accum;
    uint32_t tmem_base;
    int abort;
};

// Block-scaled MMA instruction descriptor: A and B E2M1 (format code 1 of
// the mxf4 kinds), both K-major, N/8 at bit 17, scale type UE4M3 (bit 23
// clear), M/16 at bit 24, scale-factor data ids 0 (scale_vec::4X uses all
// four bytes of a column).
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                           (static_cast<uint32_t>(BM >> 4) << 24);

struct Params {
    float *dst;
    int M, N, K;
    int splits;  // CTAs per output tile (a cluster along z), each a contiguous share of the k stages
    int dtma;    // 1: the tile is stored with TMA stores through map_d (M % 4 == 0)
    uint32_t *status;
    uint64_t limit_ns;
};
}  // namespace f4

// D[tmem] (+)= A(E2M1)[smem] * B(E2M1)[smem]^T with the E4M3 block scales of
// A and B read from tensor memory (four per row per K = 64 step).
__device__ __forceinline__ void mma_fp4_block(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ bool f4_wait_drain(uint64_t *bar, uint32_t parity, uint32_t *status, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

__global__ void __launch_bounds__(f4::THREADS, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap map_wc, const __grid_constant__ CUtensorMap map_ws,
                    const __grid_constant__ CUtensorMap map_xc, const __grid_constant__ CUtensorMap map_xs,
                    const __grid_constant__ CUtensorMap map_d, const f4::Params p) {
    using namespace f4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl *ctl = reinterpret_cast<Ctl *>(base + STAGES * STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int S = p.splits;
    const int z = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int kt0 = z * (p.K / KS) / S, kt1 = (z + 1) * (p.K / KS) / S;
    const int NK = kt1 - kt0;  // this CTA's stages (>= 1)
    float *sRed = reinterpret_cast<float *>(base);  // the fp32 tile [BN][BM], after the main loop
    // stage s: [W codes][X codes][W scales][X scales]
    auto wc = [&](int s) { return base + s * STAGE; };
    auto xc = [&](int s) { return base + s * STAGE + CODE_TILE; };
    auto wsc = [&](int s) { return base + s * STAGE + 2 * CODE_TILE; };
    auto xsc = [&](int s) { return base + s * STAGE + 2 * CODE_TILE + SCALE_TILE; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->sf_full[s], 4);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->accum, 1);
        ctl->abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&map_wc);
        prefetch_tensormap(&map_ws);
        prefetch_tensormap(&map_xc);
        prefetch_tensormap(&map_xs);
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
    griddep_wait();

    if (warp == 0) {
        // ------------- TMA producer -------------
        if (lane == 0) {
            int last[STAGES];
            for (int s = 0; s < STAGES; ++s) last[s] = -1;
            for (int i = 0; i < NK; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait_bounded(&ctl->empty[s], ph ^ 1, abort, p.status, p.limit_ns)) break;
                mbar_arrive_expect_tx(&ctl->full[s], STAGE);
                const int kx = (kt0 + i) * (KS / 2), ksx = (kt0 + i) * (KS / 16);  // byte coordinates of the stage
                tma_load_2d(wc(s), &map_wc, kx, m0, &ctl->full[s]);
                tma_load_2d(xc(s), &map_xc, kx, n0, &ctl->full[s]);
                tma_load_2d(wsc(s), &map_ws, ksx, m0, &ctl->full[s]);
                tma_load_2d(xsc(s), &map_xs, ksx, n0, &ctl->full[s]);
                last[s] = i;
            }
            if (*abort) {
                for (int s = 0; s < STAGES; ++s)
                    if (last[s] >= 0) f4_wait_drain(&ctl->full[s], (last[s] / STAGES) & 1, p.status, p.limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------- MMA issuer -------------
        if (lane == 0) {
            for (int i = 0; i < NK; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait_bounded(&ctl->full[s], ph, abort, p.status, p.limit_ns)) break;
                if (!mbar_wait_bounded(&ctl->sf_full[s], ph, abort, p.status, p.limit_ns)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(wc(s)), b_addr = smem_u32(xc(s));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // K step kk: 64 values = 32 bytes into each 128-byte swizzled row
                    const uint64_t ad = sw128_desc(a_addr + 32u * kk), bd = sw128_desc(b_addr + 32u * kk);
                    const uint32_t sfa = tmem + static_cast<uint32_t>(SF_COL0 + 32 * s + 4 * kk);
                    const uint32_t sfb = tmem + static_cast<uint32_t>(SF_COL0 + 32 * s + 16 + 4 * kk);
                    mma_fp4_block(tmem, ad, bd, IDESC, sfa, sfb, (i | kk) != 0);
                }
                mma_commit(&ctl->empty[s]);
            }
            mma_commit(&ctl->accum);  // arrives once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // ------------- scale movers -------------
        const int q = warp & 3;  // lane quarter of this warp (each quarter gets the same copy)
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
        for (int i = 0; i < NK; ++i) {
            const int s = i % STAGES;
            const uint32_t ph = (i / STAGES) & 1;
            const bool ok = mbar_wait_bounded(&ctl->full[s], ph, abort, p.status, p.limit_ns);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            // full[s] also means the MMAs that last read slot s's scale
            // columns have completed (the producer waited for them first)
            // rows lane, lane+32, lane+64, lane+96: 16 scale bytes each (word kk
            // = the four k blocks of MMA kk); column 4kk + i <- row 32i + lane
            uint32_t ra[16], rb[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 a = *reinterpret_cast<const uint4 *>(wsc(s) + 16 * (32 * i + lane));
                const uint4 b = *reinterpret_cast<const uint4 *>(xsc(s) + 16 * (32 * i + lane));
                ra[i] = a.x; ra[4 + i] = a.y; ra[8 + i] = a.z; ra[12 + i] = a.w;
                rb[i] = b.x; rb[4 + i] = b.y; rb[8 + i] = b.z; rb[12 + i] = b.w;
            }
            tmem_st_32x32b_x16(tq + static_cast<uint32_t>(SF_COL0 + 32 * s), ra);
            tmem_st_32x32b_x16(tq + static_cast<uint32_t>(SF_COL0 + 32 * s + 16), rb);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->sf_full[s]);
        }
    }

    // ---------------- epilogue (warps 2-5) ----------------
    // The fp32 tile goes through shared memory as [BN][BM] (m contiguous; the
    // stage ring is free once every MMA has completed), a TMA store for each
    // 32 columns as soon as the four warps have written them;
    // with split-K the CTAs of a cluster each sum a column slice of all the
    // partial tiles in rank order through distributed shared memory.
    const bool is_epi = warp >= 2;
    bool have = false;
    if (is_epi) {
        const bool drained = f4_wait_drain(&ctl->accum, 0, p.status, p.limit_ns);
        if (warp == 2 && lane == 0) griddep_launch();
        if (!drained) *abort = 1;
        have = __all_sync(0xFFFFFFFFu, drained && !*abort);
        if (have) tc_fence_after();
        const int q = warp & 3;
        const int r = 32 * q + lane;  // tile row (m)
        const bool pipe = S == 1 && p.dtma;  // store each 32-column group as soon as it is in shared memory
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            if (have) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * c, v);
                tmem_ld_wait();
#pragma unroll
                for (int j2 = 0; j2 < 32; ++j2) sRed[(32 * c + j2) * BM + r] = __uint_as_float(v[j2]);
            }
            if (pipe) {
                fence_proxy_async_smem();
                asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
                if (warp == 2 && lane == 0 && !*abort) {
                    tma_store_2d(&map_d, m0, n0 + 32 * c, sRed + 32 * c * BM);
                    bulk_commit_group();
                }
            }
        }
        if (pipe && warp == 2 && lane == 0 && !*abort) bulk_wait_group_read0();
    } else if (threadIdx.x == 0) {
        griddep_launch();
    }
    if (S == 1) {
        if (is_epi) {
            fence_proxy_async_smem();  // the generic-proxy writes above, before the TMA store reads them
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (p.dtma) {
                // stored group by group above
            } else if (!*abort) {
                const int et = threadIdx.x - 64;  // 0..127
                for (int it = et; it < BN * BM; it += 128) {
                    const int cl = it / BM, rr = it % BM;
                    const int gn = n0 + cl, gm = m0 + rr;
                    if (gn < p.N && gm < p.M) p.dst[static_cast<int64_t>(gn) * p.M + gm] = sRed[cl * BM + rr];
                }
            }
        }
    } else {
        __syncwarp();
        cluster_sync_all();
        int any_abort = 0;
        for (int pr = 0; pr < S; ++pr) any_abort |= ld_dsmem_u32(mapa_shared(smem_u32(&ctl->abort), pr));
        splitk_reduce_store<BM>(smem_u32(sRed), S, z, BN, m0, n0, p.M, p.N, p.dst, static_cast<int>(threadIdx.x),
                                   THREADS, any_abort != 0);
        __syncwarp();
        cluster_arrive_relaxed_wait();  // peers keep their partials until every slice is read
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Activation rows -> NVFP4 V2 rows: per block of 16, scale = the E4M3 value
// nearest amax/6 (round to nearest even, saturating), codes = the E2M1 value
// nearest x/scale (the same), both decided in float32 by the hardware
// conversions; zero codes when the scale is zero.  One thread per block.
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const float *__restrict__ x, uint8_t *__restrict__ out,
                                                             int64_t rows, int64_t k) {
    griddep_wait();
    griddep_launch();
    const int64_t nb = k / 16, total = rows * nb, rb = k / 32 * 18;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total; t += stride) {
        const int64_t r = t / nb, b = t - r * nb;
        const float4 *src = reinterpret_cast<const float4 *>(x + r * k + 16 * b);
        float v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 a = __ldg(src + i);
            v[4 * i] = a.x;
            v[4 * i + 1] = a.y;
            v[4 * i + 2] = a.z;
            v[4 * i + 3] = a.w;
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
        const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(__fdiv_rn(amax, 6.0f), __NV_SATFINITE, __NV_E4M3);
        const float s = e4m3_to_f32(sc);
        uint32_t w0 = 0, w1 = 0;
        if (s != 0.0f) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t c = __nv_cvt_float_to_fp4(__fdiv_rn(v[j], s), __NV_E2M1, cudaRoundNearest) & 15u;
                if (j < 8)
                    w0 |= c << (4 * j);
                else
                    w1 |= c << (4 * (j - 8));
            }
        }
        uint8_t *row = out + r * rb;
        *reinterpret_cast<uint2 *>(row + 8 * b) = make_uint2(w0, w1);
        row[k / 2 + b] = sc;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 f4_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D byte map over `rows` rows of `width` bytes at `ptr` with row pitch
// `pitch`, box [box_rows][box_w] bytes, optional 128-byte swizzle; zero fill.
bool f4_map(CUtensorMap *map, const void *ptr, int64_t width, int64_t rows, int64_t pitch, int box_w, int box_rows,
            bool swizzle) {
    auto fn = f4_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_w), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t gemm_fp4_init() {
    return cudaFuncSetAttribute(gemm_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(f4::SMEM));
}

cudaError_t launch_quantize_nvfp4(const float *x, void *out, int64_t rows, int64_t k, int num_sms, cudaStream_t st) {
    const int64_t total = rows * (k / 16);
    const int64_t want = (total + 255) / 256;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 4LL * num_sms)));
    return launch_pdl(quantize_nvfp4_kernel, dim3(grid), dim3(256), 0, st, dim3(1, 1, 1), x,
                      static_cast<uint8_t *>(out), rows, k);
}

cudaError_t launch_gemm_fp4(const void *w, const void *xq, float *dst, int64_t m, int64_t k, int64_t n, int num_sms,
                            uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    using namespace f4;
    const int64_t rb = k / 32 * 18;  // V2 row bytes of W and of Xq
    CUtensorMap mwc, mws, mxc, mxs;
    const uint8_t *wb = static_cast<const uint8_t *>(w), *xb = static_cast<const uint8_t *>(xq);
    if (!f4_map(&mwc, wb, k / 2, m, rb, 128, BM, true) || !f4_map(&mws, wb + k / 2, k / 16, m, rb, 16, BM, false) ||
        !f4_map(&mxc, xb, k / 2, n, rb, 128, BN, true) || !f4_map(&mxs, xb + k / 2, k / 16, n, rb, 16, BN, false))
        return cudaErrorInvalidValue;
    Params p;
    p.dst = dst;
    p.M = static_cast<int>(m);
    p.N = static_cast<int>(n);
    p.K = static_cast<int>(k);
    p.status = status;
    p.limit_ns = limit_ns;
    // split-K: enough CTAs per tile to cover the SMs, at most one per stage,
    // a power of two up to 8 (it divides the tile width)
    const int64_t tiles = ((m + BM - 1) / BM) * ((n + BN - 1) / BN);
    int sp = 1;
    while (sp < 8 && tiles * (sp * 2) <= num_sms && sp * 2 <= k / KS) sp *= 2;
    p.splits = sp;
    // dst [n][m] f32 as a TMA store target: boxes of [BN n][BM m]
    CUtensorMap mdst;
    memset(&mdst, 0, sizeof(mdst));
    p.dtma = 0;
    if (m % 4 == 0) {
        auto fn = f4_encode_fn();
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(m), static_cast<cuuint64_t>(n)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(m) * 4};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(BM), 32u};
        const cuuint32_t estr[2] = {1, 1};
        p.dtma = fn && fn(&mdst, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dst, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const dim3 grid(static_cast<unsigned>((m + BM - 1) / BM), static_cast<unsigned>((n + BN - 1) / BN),
                    static_cast<unsigned>(sp));
    return launch_pdl(gemm_fp4_kernel, grid, dim3(THREADS), SMEM, st, dim3(1, 1, static_cast<unsigned>(sp)), mwc,
                      mws, mxc, mxs, mdst, p);
}

}  // namespace qmm
