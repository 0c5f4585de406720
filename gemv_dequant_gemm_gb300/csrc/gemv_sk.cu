// gemv_sk.cu -- the small-batch GEMV (1 <= n <= 8) for short calls: many
// small CTAs, X in registers, k split across a thread-block cluster.
//
// The product is the batched GEMV of aprender-serve 0.70.2
// cublas_prefill/mod.rs (doc comment of cublas_gemm_threshold, which names
// the "insufficient parallelism" of a one-warp-per-row Q4K GEMV at M <= 8):
//     dst[i][row] = sum_c W[row][c] * X[i][c].
// A few megabytes of weights are streamed once, so a call is bound by
// latency, not bandwidth: the design spreads the work over every SM with
// enough resident warps to hide it, and keeps the per-weight instruction
// count low.
//
//   * A CTA owns up to RB consecutive rows (the rows spread evenly over a
//     grid of whole waves per SM when one wave holds it) and one k-slice of
//     them: a split S of a cluster of S CTAs along k, S = 1 (whole rows)
//     unless that leaves too few warps to cover the SMs.  n > 4 (or n > 2
//     when that avoids a k split) spreads the activation rows over several
//     CTAs.  Thread 0 moves the rows' slice bytes into
//     shared memory with bulk copies (one copy when the slice is the whole
//     row, one per row otherwise; 16-byte aligned supersets, any row stride)
//     after warming L2 with them before the dependency wait.
//   * Once the bytes are in, the scale (and Q4_K minimum) of every scale
//     region of the CTA's rows is decoded once into shared memory.
//   * Thread t owns the 8-weight units t, t + TK, ... (J of them) of the
//     slice and keeps X at those k positions for all n rows in registers, as
//     f32 pairs (J * 8 * n floats), loaded once.  Per W row it turns each
//     unit's codes into exact f32 pairs (a byte under the exponent of 2^23
//     and one paired subtraction; NVFP4 by the hardware E2M1 conversion),
//     multiplies them with paired FMAs, and scales the unit's sum once; rows
//     are taken four (n > 4: two) at a time and reduced across each warp with
//     a butterfly that leaves value i in lane i.
//   * The warps' partials are added in warp order; with S > 1 each CTA then
//     sums a share of the RB x n results over the cluster's S partial tiles
//     through distributed shared memory, in rank order.  No atomics: the
//     result is deterministic.  The fp32 chains are short (8 weights per
//     unit, a few units per thread, a 5-level shuffle tree, S ranks), so the
//     rounding error stays far below 1e-5 * sum|W*X|.
//   * The one wait (for the weight copies) is bounded; when it runs out the
//     CTA latches the timeout bit, stores nothing, keeps to the cluster
//     barriers and waits for its copies before it exits.
#include <algorithm>
#include <atomic>

#include "decode.cuh"
#include "kernels.h"
#include "l2hint.cuh"

namespace qmm {

namespace gs {
constexpr int UW = 8;            // weights per unit
constexpr int RG = 4;            // rows per reduction group
constexpr int MAX_THREADS = 256;
constexpr int MAX_RB = 32;
constexpr int SMEM_CAP = 96 * 1024;

struct Params {
    const uint8_t *w;
    const float *x;
    float *dst;
    int64_t rb, k;
    int m, n;
    int nvc;          // activation rows per CTA (grid z splits n when n > 4)
    int splits;       // S: CTAs of a cluster along k (grid y)
    int us;           // units per split
    int rbk;          // RB: rows per CTA (a multiple of RG)
    int slice_bytes;  // bytes of one row's k-slice
    int pitch;        // shared-memory row pitch when S > 1
    int wbuf_bytes;   // shared bytes for the weights
    uint32_t *status;
    uint64_t limit_ns;
};

template <int NV> constexpr int nvp() { return NV <= 1 ? 1 : (NV <= 2 ? 2 : (NV <= 4 ? 4 : 8)); }
}  // namespace gs

// ---- per-format pieces: scale regions and the exact codes of 8 weights ----

template <int F> struct SkFmt;
template <> struct SkFmt<QMM_Q4_0> { static constexpr int RS = 32, NSC = 1; };
template <> struct SkFmt<QMM_Q8_0> { static constexpr int RS = 32, NSC = 1; };
template <> struct SkFmt<QMM_Q4_K> { static constexpr int RS = 32, NSC = 2; };  // scale and minimum
template <> struct SkFmt<QMM_Q6_K> { static constexpr int RS = 16, NSC = 1; };
template <> struct SkFmt<QMM_NVFP4> { static constexpr int RS = 16, NSC = 1; };

// 4 bytes from a 2-byte aligned shared address
__device__ __forceinline__ uint32_t sk_ld16x2(const uint8_t *p) {
    const uint16_t *q = reinterpret_cast<const uint16_t *>(p);
    return static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 16);
}

// Bytes j and j+1 of w (each a small unsigned code) as floats minus `bias`,
// exactly: the byte goes under the exponent of 2^23, then one paired add.
__device__ __forceinline__ uint64_t sk_byte_pair(uint32_t w, int j, uint64_t minus) {
    const float a = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | static_cast<uint32_t>(j)));
    const float b = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | static_cast<uint32_t>(j + 1)));
    return f2_add(f2_pack(a, b), minus);
}

__device__ __forceinline__ void sk_words_to_pairs(uint32_t lo, uint32_t hi, float bias, uint64_t (&w)[4]) {
    const float mb = -(8388608.0f + bias);
    const uint64_t minus = f2_pack(mb, mb);
    w[0] = sk_byte_pair(lo, 0, minus);
    w[1] = sk_byte_pair(lo, 2, minus);
    w[2] = sk_byte_pair(hi, 0, minus);
    w[3] = sk_byte_pair(hi, 2, minus);
}

// The exact code values of weights e0..e0+7 (e0 % 8 == 0) of the row at rowp,
// as 4 f32 pairs in k order; the region scale is applied by the caller.
template <int F> __device__ __forceinline__ void sk_unit8(const uint8_t *rowp, int64_t e0, uint64_t (&w)[4]);

template <> __device__ __forceinline__ void sk_unit8<QMM_Q4_0>(const uint8_t *rowp, int64_t e0, uint64_t (&w)[4]) {
    const int e = static_cast<int>(e0 & 31);
    const uint8_t *q = rowp + (e0 >> 5) * 18 + 2 + (e & 15);
    uint32_t lo = sk_ld16x2(q), hi = sk_ld16x2(q + 4);
    if (e >= 16) {
        lo >>= 4;
        hi >>= 4;
    }
    sk_words_to_pairs(lo & 0x0F0F0F0Fu, hi & 0x0F0F0F0Fu, 8.0f, w);  // q - 8
}

template <> __device__ __forceinline__ void sk_unit8<QMM_Q8_0>(const uint8_t *rowp, int64_t e0, uint64_t (&w)[4]) {
    const uint8_t *q = rowp + (e0 >> 5) * 34 + 2 + (e0 & 31);
    sk_words_to_pairs(sk_ld16x2(q) ^ 0x80808080u, sk_ld16x2(q + 4) ^ 0x80808080u, 128.0f, w);  // (q + 128) - 128
}

template <> __device__ __forceinline__ void sk_unit8<QMM_Q4_K>(const uint8_t *rowp, int64_t e0, uint64_t (&w)[4]) {
    const int e = static_cast<int>(e0 & 255);
    const int c = e >> 6, r = e & 63;
    uint2 q = *reinterpret_cast<const uint2 *>(rowp + (e0 >> 8) * 144 + 16 + 32 * c + (r & 31));
    if (r >= 32) {
        q.x >>= 4;
        q.y >>= 4;
    }
    sk_words_to_pairs(q.x & 0x0F0F0F0Fu, q.y & 0x0F0F0F0Fu, 0.0f, w);  // q (the minimum is a separate term)
}

template <> __device__ __forceinline__ void sk_unit8<QMM_Q6_K>(const uint8_t *rowp, int64_t e0, uint64_t (&w)[4]) {
    const uint8_t *blk = rowp + (e0 >> 8) * 210;
    const int e = static_cast<int>(e0 & 255);
    const int h = e >> 7, s = (e & 127) >> 5, l = e & 31;
    const uint8_t *ql = blk + 64 * h + l + 32 * (s & 1);
    const uint8_t *qh = blk + 128 + 32 * h + l;
    const int lsh = (s >= 2) ? 4 : 0, hsh = 2 * s;
    const uint32_t q0 = ((sk_ld16x2(ql) >> lsh) & 0x0F0F0F0Fu) | (((sk_ld16x2(qh) >> hsh) & 0x03030303u) << 4);
    const uint32_t q1 = ((sk_ld16x2(ql + 4) >> lsh) & 0x0F0F0F0Fu) | (((sk_ld16x2(qh + 4) >> hsh) & 0x03030303u) << 4);
    sk_words_to_pairs(q0, q1, 32.0f, w);  // q - 32
}

template <> __device__ __forceinline__ void sk_unit8<QMM_NVFP4>(const uint8_t *rowp, int64_t e0, uint64_t (&w)[4]) {
    const int e = static_cast<int>(e0 & 63);
    e2m1x8_to_f2(*reinterpret_cast<const uint32_t *>(rowp + (e0 >> 6) * 36 + 4 + (e >> 1)), w);
}

// Scale (and Q4_K minimum) of scale region `reg` (RS weights) of a row.
template <int F> __device__ __forceinline__ void sk_region_scale(const uint8_t *rowp, int64_t reg, float &s, float &o) {
    o = 0.0f;
    if constexpr (F == QMM_Q4_0 || F == QMM_Q8_0) {
        s = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(rowp + reg * (F == QMM_Q4_0 ? 18 : 34)));
    } else if constexpr (F == QMM_Q4_K) {
        const uint8_t *blk = rowp + (reg >> 3) * 144;
        const int j = static_cast<int>(reg & 7);
        const uint16_t *dd = reinterpret_cast<const uint16_t *>(blk);
        const uint8_t *sc12 = blk + 4;
        int sc, mn;
        if (j < 4) {
            sc = sc12[j] & 63;
            mn = sc12[j + 4] & 63;
        } else {
            sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
            mn = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
        }
        s = __fmul_rn(half_bits_to_f32(dd[0]), static_cast<float>(sc));
        o = __fmul_rn(half_bits_to_f32(dd[1]), static_cast<float>(mn));
    } else if constexpr (F == QMM_Q6_K) {
        const uint8_t *blk = rowp + (reg >> 4) * 210;
        s = __fmul_rn(half_bits_to_f32(*reinterpret_cast<const uint16_t *>(blk + 208)),
                      static_cast<float>(static_cast<int8_t>(blk[192 + (reg & 15)])));
    } else {  // NVFP4
        s = e4m3_to_f32(rowp[(reg >> 2) * 36 + (reg & 3)]);
    }
}

template <int F, int NV, int J>
__global__ void __launch_bounds__(gs::MAX_THREADS) gemv_sk_kernel(const gs::Params p) {
    using namespace gs;
    constexpr int QK = Fmt<F>::QK, BB = Fmt<F>::BB;
    constexpr int RS = SkFmt<F>::RS, NSC = SkFmt<F>::NSC;
    constexpr int NVP = nvp<NV>();
    constexpr int RGV = RG;                 // rows per butterfly
    constexpr int V = RGV * NVP;            // values one butterfly reduces (<= 32)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *wbuf = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int tk = blockDim.x, nwarps = tk >> 5;
    const int nsr = p.us * UW / RS;                                 // scale regions per row slice
    float *scl = reinterpret_cast<float *>(wbuf + p.wbuf_bytes);    // [RB][nsr][NSC]
    float *part = scl + p.rbk * nsr * NSC;                          // [nwarps][RB * NVP]
    float *red = part + nwarps * p.rbk * NVP;                       // [NV][RB]
    uint64_t *bar = reinterpret_cast<uint64_t *>(red + ((p.rbk * NV + 1) & ~1));
    int *abort_flag = reinterpret_cast<int *>(bar + 1);  // nonzero: this CTA's wait ran out (read by the cluster)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.splits;
    const int z = blockIdx.y;  // rank in the cluster (cluster dims 1 x S x 1, grid y = S)
    // rows spread evenly over the grid (at most p.rbk per CTA)
    const int row0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.m / gridDim.x);
    const int rows = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.m / gridDim.x) - row0;
    const int64_t kb0 = static_cast<int64_t>(z) * p.us * UW;  // first k of the slice
    const int64_t sbo = kb0 / QK * BB;                         // its byte offset in a row
    const uintptr_t wbase = reinterpret_cast<uintptr_t>(p.w);

    if (tid == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        // a cache hint, harmless whatever the kernel in front is writing
        if (S == 1) {
            prefetch_l2_range(wbase + static_cast<uintptr_t>(row0 * p.rb),
                              wbase + static_cast<uintptr_t>((row0 + rows) * p.rb));
        } else {
            for (int r = 0; r < rows; ++r) {
                const uintptr_t a = wbase + static_cast<uintptr_t>((row0 + r) * p.rb + sbo);
                prefetch_l2_range(a, a + p.slice_bytes);
            }
        }
    }
    __syncthreads();
    griddep_wait();
    if (tid == 0) {
        if (S == 1) {  // the rows are contiguous: one copy
            const uintptr_t src = wbase + static_cast<uintptr_t>(row0 * p.rb);
            const uintptr_t a = src & ~uintptr_t(15);
            const uint32_t len = (static_cast<uint32_t>(src - a) + static_cast<uint32_t>(rows * p.rb) + 15u) & ~15u;
            mbar_arrive_expect_tx(bar, len);
            bulk_load_1d(wbuf, reinterpret_cast<const void *>(a), len, bar);
        } else {
            uint32_t tot = 0;
            for (int r = 0; r < rows; ++r) {
                const uintptr_t src = wbase + static_cast<uintptr_t>((row0 + r) * p.rb + sbo);
                tot += (static_cast<uint32_t>(src & 15u) + static_cast<uint32_t>(p.slice_bytes) + 15u) & ~15u;
            }
            mbar_arrive_expect_tx(bar, tot);
            for (int r = 0; r < rows; ++r) {
                const uintptr_t src = wbase + static_cast<uintptr_t>((row0 + r) * p.rb + sbo);
                const uintptr_t a = src & ~uintptr_t(15);
                const uint32_t len = (static_cast<uint32_t>(src - a) + static_cast<uint32_t>(p.slice_bytes) + 15u) & ~15u;
                bulk_load_1d(wbuf + r * p.pitch, reinterpret_cast<const void *>(a), len, bar);
            }
        }
        griddep_launch();
    }

    // X at this thread's k positions, for this CTA's activation rows
    // v0 .. v0 + nv - 1, as f32 pairs
    const int v0 = blockIdx.z * p.nvc;
    const int nv = min(p.nvc, p.n - v0);
    uint64_t x2[J][NV][4];
    float xs[J][NV];  // per-unit sums of X (the Q4_K minimum term)
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int u = tid + tk * j;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (u < p.us && v < nv) {
                const float4 *src =
                    reinterpret_cast<const float4 *>(p.x + static_cast<int64_t>(v0 + v) * p.k + kb0 + u * UW);
                a = __ldg(src);
                b = __ldg(src + 1);
            }
            x2[j][v][0] = f2_pack(a.x, a.y);
            x2[j][v][1] = f2_pack(a.z, a.w);
            x2[j][v][2] = f2_pack(b.x, b.y);
            x2[j][v][3] = f2_pack(b.z, b.w);
            xs[j][v] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
        }
    }
    const bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0, abort_flag, p.status, p.limit_ns)) != 0;

    // row pointer such that rowp + (e0/QK)*BB is the block of weight e0
    auto row_ptr = [&](int rl) -> const uint8_t * {
        if (S == 1) return wbuf + ((wbase + static_cast<uintptr_t>(row0 * p.rb)) & 15u) + rl * p.rb;
        return wbuf + rl * p.pitch + ((wbase + static_cast<uintptr_t>((row0 + rl) * p.rb + sbo)) & 15u) - sbo;
    };
    if (ok) {
        // every region's scale once, into shared memory
        const int64_t reg0 = kb0 / RS;
        for (int i = tid; i < rows * nsr; i += tk) {
            const int rl = i / nsr, s = i - rl * nsr;
            float sc, of;
            sk_region_scale<F>(row_ptr(rl), reg0 + s, sc, of);
            scl[i * NSC] = sc;
            if constexpr (NSC == 2) scl[i * NSC + 1] = of;
        }
    }
    __syncthreads();
    if (ok) {
        for (int g0 = 0; g0 < rows; g0 += RGV) {  // uniform over the CTA
            uint64_t acc2[RGV][NV];  // (even, odd) k partial sums of each row and activation row
            float accm[RGV][NV];     // Q4_K: the minimum term
#pragma unroll
            for (int r = 0; r < RGV; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    acc2[r][v] = f2_pack(0.0f, 0.0f);
                    accm[r][v] = 0.0f;
                }
#pragma unroll
            for (int r = 0; r < RGV; ++r) {
                const int rl = g0 + r;
                if (rl < rows) {  // uniform
                    const uint8_t *rowp = row_ptr(rl);
                    const float *rs = scl + rl * nsr * NSC;
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const int u = tid + tk * j;
                        if (u < p.us) {
                            uint64_t w2[4];
                            sk_unit8<F>(rowp, kb0 + u * UW, w2);
                            const int ri = (u * UW) / RS;
                            const float sc = rs[ri * NSC];
                            const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
                            for (int v = 0; v < NV; ++v) {
                                uint64_t pr = f2_fma(w2[0], x2[j][v][0], f2_pack(0.0f, 0.0f));
                                pr = f2_fma(w2[1], x2[j][v][1], pr);
                                pr = f2_fma(w2[2], x2[j][v][2], pr);
                                pr = f2_fma(w2[3], x2[j][v][3], pr);
                                acc2[r][v] = f2_fma(sc2, pr, acc2[r][v]);
                                if constexpr (NSC == 2) accm[r][v] = __fmaf_rn(-rs[ri * NSC + 1], xs[j][v], accm[r][v]);
                            }
                        }
                    }
                }
            }
            float a[V];
#pragma unroll
            for (int r = 0; r < RGV; ++r)
#pragma unroll
                for (int v = 0; v < NVP; ++v) {
                    if (v < NV) {
                        const float2 h = f2_unpack(acc2[r][v]);
                        a[r * NVP + v] = (h.x + h.y) + accm[r][v];
                    } else {
                        a[r * NVP + v] = 0.0f;
                    }
                }
            const float s = warp_transpose_sum<V>(a, lane);
            if (lane < V) part[warp * (p.rbk * NVP) + g0 * NVP + lane] = s;
        }
    }
    __syncthreads();
    // the warps' partials in warp order; element e = v * RB + r
    for (int e = tid; e < NV * p.rbk; e += tk) {
        const int v = e / p.rbk, r = e - v * p.rbk;
        float s = 0.0f;
        for (int w = 0; w < nwarps; ++w) s += part[w * (p.rbk * NVP) + r * NVP + v];
        if (S == 1) {
            if (ok && r < rows && v < nv) p.dst[static_cast<int64_t>(v0 + v) * p.m + row0 + r] = s;
        } else {
            red[e] = s;
        }
    }
    if (S > 1) {
        // every CTA of the cluster reaches both barriers, whatever its wait did
        __syncthreads();
        cluster_sync_all();
        int any_bad = 0;
        for (int pr = 0; pr < S; ++pr) any_bad |= ld_dsmem_u32(mapa_shared(smem_u32(abort_flag), pr));
        if (!any_bad) {
            for (int e = z + S * tid; e < NV * p.rbk; e += S * tk) {
                const int v = e / p.rbk, r = e - v * p.rbk;
                if (r < rows && v < nv) {
                    float s = 0.0f;
                    for (int pr = 0; pr < S; ++pr) s += ld_dsmem_f32(mapa_shared(smem_u32(red + e), pr));
                    p.dst[static_cast<int64_t>(v0 + v) * p.m + row0 + r] = s;
                }
            }
        }
        cluster_arrive_relaxed_wait();  // peers keep their partials until every share is read
    }
    if (!ok && tid == 0) {  // copies still in flight land before the CTA exits
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar, 0) && global_timer_ns() - t0 < p.limit_ns) {
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

struct SkPlan {
    int splits, us, tk, J, rbk;
};

// Shared bytes of an instance: weights, region scales, warp partials, the
// reduced tile, barrier and flag.
size_t sk_smem(int wbuf_bytes, int rbk, int us, int rs, int nsc, int tk, int nvp_, int nv) {
    return 128 + static_cast<size_t>(wbuf_bytes) + static_cast<size_t>(rbk) * (us * gs::UW / rs) * nsc * 4 +
           static_cast<size_t>(tk / 32) * rbk * nvp_ * 4 + static_cast<size_t>((rbk * nv + 1) & ~1) * 4 + 16;
}

// Splits S (the slice a whole number of blocks), threads TK and units per
// thread J (X registers J*8*n <= 64), rows per CTA RB: the fewest splits that
// give the GPU about twelve resident warps per SM; RB sized below.
bool plan_sk(int qk, int bb, int64_t m, int64_t k, int nv, int nz, int jcap, int num_sms, SkPlan &pl) {
    using namespace gs;
    if (k % UW != 0 || m < 1) return false;
    const int64_t U = k / UW;
    const int jmax = std::max(1, std::min(jcap, 64 / (UW * nv)));
    bool have = false;
    int64_t best_warps = -1;
    for (int S = 1; S <= 8; ++S) {
        if (U % S != 0) continue;
        const int64_t us = U / S;
        if ((us * UW) % qk != 0) continue;
        int best_tk = 0;
        int64_t best_waste = INT64_MAX;
        for (int tk = 32; tk <= MAX_THREADS; tk += 32) {
            const int64_t J = (us + tk - 1) / tk;
            if (J > jmax) continue;
            if (tk < 64 && us >= 64) continue;  // at least two warps when the slice allows
            const int64_t waste = tk * J - us;
            // among equal waste: with one activation row per CTA, more units
            // per thread (more independent work for the same registers);
            // with more, more threads (measured on GB300)
            const bool better_tie = nv == 1 ? tk < best_tk : tk > best_tk;
            if (waste < best_waste || (waste == best_waste && better_tie)) {
                best_waste = waste;
                best_tk = tk;
            }
        }
        if (best_tk == 0) continue;
        const int64_t warps = (m + RG - 1) / RG * S * (best_tk / 32) * nz;
        if (!have || warps > best_warps) {
            have = true;
            best_warps = warps;
            pl.splits = S;
            pl.us = static_cast<int>(us);
            pl.tk = best_tk;
            pl.J = static_cast<int>((us + best_tk - 1) / best_tk);
        }
        if (warps >= static_cast<int64_t>(num_sms) * 8) break;  // the fewest splits that fill the GPU
    }
    if (!have) return false;
    // rows per CTA for about 16 resident warps per SM when a thread holds one
    // or two activation rows, 32 with more (measured on GB300)
    const int64_t work = m * pl.splits * (pl.tk / 32) * nz;
    const int64_t warps_per_sm = nv <= 2 ? 16 : 32;
    int64_t rb = (work / (static_cast<int64_t>(num_sms) * warps_per_sm) + RG / 2) / RG * RG;
    rb = std::max<int64_t>(RG, std::min<int64_t>(MAX_RB, rb));
    rb = std::min<int64_t>(rb, (m + RG - 1) / RG * RG);
    const int64_t slice = static_cast<int64_t>(pl.us) * UW / qk * bb;
    // shared memory: weights, warp partials, the reduced tile, barrier
    auto smem_of = [&](int64_t r) {
        const int64_t wb = pl.splits == 1 ? (r * (k / qk * bb) + 15 + 15) / 16 * 16 : r * ((slice + 15 + 15) / 16 * 16);
        return static_cast<int64_t>(sk_smem(static_cast<int>(wb), static_cast<int>(r), pl.us, 16, 2, pl.tk, 8, 8));
    };
    while (rb > RG && smem_of(rb) > SMEM_CAP) rb -= RG;
    if (smem_of(rb) > SMEM_CAP) return false;
    pl.rbk = static_cast<int>(rb);
    return true;
}

template <int F, int NV, int J> cudaError_t launch_sk_j(gs::Params p, SkPlan pl, int num_sms, cudaStream_t st) {
    using namespace gs;
    auto wbuf_of = [&](int rbk) {
        return pl.splits == 1 ? static_cast<int>((rbk * p.rb + 15 + 15) / 16 * 16) : rbk * p.pitch;
    };
    auto smem_of = [&](int rbk) {
        return sk_smem(wbuf_of(rbk), rbk, pl.us, SkFmt<F>::RS, SkFmt<F>::NSC, pl.tk, nvp<NV>(), NV);
    };
    // Resident CTAs per SM of this instance at this size (registers usually
    // decide); cached per instance, a 64-bit word (block size, shared bytes,
    // result) so concurrent callers read a consistent entry.
    static std::atomic<uint64_t> cache{0};
    auto resident = [&](int tk, size_t smem) -> int {
        const uint64_t key = (static_cast<uint64_t>(tk) << 48) | (static_cast<uint64_t>(smem) << 16);
        const uint64_t c = cache.load(std::memory_order_relaxed);
        if ((c & ~uint64_t(0xFFFF)) == key) return static_cast<int>(c & 0xFFFF);
        int occ = 0;
        if (cudaFuncSetAttribute(gemv_sk_kernel<F, NV, J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_sk_kernel<F, NV, J>, tk, smem) != cudaSuccess)
            return 0;
        cache.store(key | static_cast<uint64_t>(occ & 0xFFFF), std::memory_order_relaxed);
        return occ;
    };
    // grow the row blocks until the grid fits in one wave of resident CTAs
    const int nz = (p.n + p.nvc - 1) / p.nvc;
    for (;;) {
        const int occ = resident(pl.tk, smem_of(pl.rbk));
        if (occ <= 0) return cudaErrorInvalidValue;
        const int64_t ctas = static_cast<int64_t>((p.m + pl.rbk - 1) / pl.rbk) * pl.splits * nz;
        if (ctas <= static_cast<int64_t>(occ) * num_sms || pl.rbk + RG > MAX_RB ||
            smem_of(pl.rbk + RG) > static_cast<size_t>(SMEM_CAP))
            break;
        pl.rbk += RG;
    }
    p.rbk = pl.rbk;
    p.wbuf_bytes = wbuf_of(pl.rbk);
    const size_t smem = smem_of(pl.rbk);
    cudaError_t e = cudaFuncSetAttribute(gemv_sk_kernel<F, NV, J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // a grid that gives every SM the same number of CTAs when one wave still
    // holds it (rows then spread evenly, at most rbk per CTA)
    int64_t gx = (p.m + pl.rbk - 1) / pl.rbk;
    {
        const int occ = resident(pl.tk, smem);
        const int64_t per = static_cast<int64_t>(pl.splits) * nz;
        int64_t g2 = gx;
        while ((g2 * per) % num_sms != 0) ++g2;
        if (g2 <= p.m && g2 * per <= static_cast<int64_t>(occ) * num_sms) gx = g2;
    }
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(pl.splits), static_cast<unsigned>(nz));
    return launch_pdl(gemv_sk_kernel<F, NV, J>, grid, dim3(pl.tk), smem, st, dim3(1, pl.splits, 1), p);
}

template <int F, int NV> cudaError_t launch_sk_nv(const gs::Params &p, const SkPlan &pl, int num_sms,
                                                  cudaStream_t st) {
    constexpr int JM = std::max(1, std::min(4, 64 / (gs::UW * NV)));
    switch (pl.J) {
    case 1: return launch_sk_j<F, NV, 1>(p, pl, num_sms, st);
    case 2: if constexpr (JM >= 2) return launch_sk_j<F, NV, 2>(p, pl, num_sms, st); else return cudaErrorInvalidValue;
    case 3: if constexpr (JM >= 3) return launch_sk_j<F, NV, 3>(p, pl, num_sms, st); else return cudaErrorInvalidValue;
    case 4: if constexpr (JM >= 4) return launch_sk_j<F, NV, 4>(p, pl, num_sms, st); else return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

template <int F> cudaError_t launch_sk_f(const gs::Params &p, const SkPlan &pl, int num_sms, cudaStream_t st) {
    switch (p.nvc) {
    case 1: return launch_sk_nv<F, 1>(p, pl, num_sms, st);
    case 2: return launch_sk_nv<F, 2>(p, pl, num_sms, st);
    case 3: return launch_sk_nv<F, 3>(p, pl, num_sms, st);
    case 4: return launch_sk_nv<F, 4>(p, pl, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// The split-K register-X GEMV when it has a plan for this problem: returns
// cudaErrorNotSupported (and launches nothing) when it does not.
cudaError_t launch_gemv_sk(int dtype, const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k,
                           int n, int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    int qk = 0, bb = 0;
    switch (dtype) {
    case QMM_Q4_0: qk = 32; bb = 18; break;
    case QMM_Q8_0: qk = 32; bb = 34; break;
    case QMM_Q4_K: qk = 256; bb = 144; break;
    case QMM_Q6_K: qk = 256; bb = 210; break;
    case QMM_NVFP4: qk = 64; bb = 36; break;
    default: return cudaErrorNotSupported;
    }
    if (n < 1 || n > 8 || m > (int64_t(1) << 30) || (reinterpret_cast<uintptr_t>(x) & 15u) != 0) return cudaErrorNotSupported;
    // n > 4: two CTAs share the activation rows (at most 4 rows of X per thread)
    int nz = n > 4 ? 2 : 1;
    int nvc = (n + nz - 1) / nz;
    SkPlan pl;
    if (!plan_sk(qk, bb, m, k, nvc, nz, 4, num_sms, pl)) return cudaErrorNotSupported;
    // a plan that splits k costs a cluster reduction; when two activation rows
    // per CTA (fewer X registers, so longer slices) avoid the split, take
    // that one (measured on GB300: 1024 x 4608, n = 4 and 8, 12-27 % faster)
    if (pl.splits > 1 && nvc > 2) {
        SkPlan p2;
        const int nz2 = (n + 1) / 2;
        if (plan_sk(qk, bb, m, k, 2, nz2, 4, num_sms, p2) && p2.splits == 1) {
            pl = p2;
            nz = nz2;
            nvc = 2;
        }
    }
    gs::Params p = {};
    p.w = static_cast<const uint8_t *>(w);
    p.x = x;
    p.dst = dst;
    p.rb = rb;
    p.k = k;
    p.m = static_cast<int>(m);
    p.n = n;
    p.nvc = nvc;
    p.splits = pl.splits;
    p.us = pl.us;
    p.rbk = pl.rbk;
    p.slice_bytes = static_cast<int>(static_cast<int64_t>(pl.us) * gs::UW / qk * bb);
    p.pitch = (p.slice_bytes + 15 + 15) / 16 * 16;
    p.wbuf_bytes = pl.splits == 1 ? static_cast<int>((pl.rbk * rb + 15 + 15) / 16 * 16) : pl.rbk * p.pitch;
    p.status = status;
    p.limit_ns = limit_ns;
    switch (dtype) {
    case QMM_Q4_0: return launch_sk_f<QMM_Q4_0>(p, pl, num_sms, st);
    case QMM_Q8_0: return launch_sk_f<QMM_Q8_0>(p, pl, num_sms, st);
    case QMM_Q4_K: return launch_sk_f<QMM_Q4_K>(p, pl, num_sms, st);
    case QMM_Q6_K: return launch_sk_f<QMM_Q6_K>(p, pl, num_sms, st);
    case QMM_NVFP4: return launch_sk_f<QMM_NVFP4>(p, pl, num_sms, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace qmm
