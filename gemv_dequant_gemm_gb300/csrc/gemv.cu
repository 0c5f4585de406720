// gemv.cu -- the small-batch GEMV (1 <= n <= 8) and the MoE gate/up GEMV.
//
// dst[i][row] = sum_c W[row][c] * X[i][c], read straight from the packed
// weights at their packed size, as the batched GEMV described in
// aprender-serve 0.70.2 cublas_prefill/mod.rs does (doc comment of
// cublas_gemm_threshold, which also names that GEMV's one-warp blocks as its
// weakness).  The MoE kernel is the served gate/up GEMV of memra-engine
// 0.128.0 moe_rows_ceiling_bench.rs: the same product over a device table of
// 2*n_pairs (plane, pair) matrices, each scaled by its own fp32 factor.
//
// Design: the rows of all matrices are cut into stages of RT consecutive
// rows.  A stage's packed bytes are contiguous in memory, so one producer
// thread moves each stage into a shared-memory ring with a single 1-D bulk
// copy (TMA) -- a 16-byte aligned superset of the rows, for any block size
// and row stride -- several stages ahead; every CTA walks a contiguous run of
// stages, so its rows stream sequentially.  Eight compute warps decode from
// shared memory and multiply by X, which is staged in shared memory once per
// CTA when it fits:
//   * rows-per-warp mode: warp w owns RPW rows of the stage and its lanes
//     split k in 8-weight groups; every X group is loaded once and reused for
//     the warp's rows;
//   * warps-per-row mode (long rows): WPR warps split one row's k range and a
//     fixed-order sum over the WPR partials finishes the row.
// Each group of 8 weights lies in one scale region of its format: its 8
// code*x products (small exact codes, grp8) are summed into a fresh partial
// that is scaled once and joins the accumulator; lanes reduce by shuffles in
// a fixed tree, so results are deterministic and the float32 rounding error
// stays far below 1e-5 * sum|W*X|.  Every wait is bounded; a stage with a
// NULL or misaligned matrix pointer is skipped, reported, and its rows set to
// NaN.
#include <algorithm>

#include "decode.cuh"
#include "kernels.h"

namespace qmm {

namespace gv {
constexpr int COMPUTE_WARPS = 8;
constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);  // + producer warp
constexpr int MAX_RING = 8;
constexpr int MAX_RPW = 4;
constexpr int SMEM_BUDGET = 226 * 1024;
constexpr int MAX_TABLE = 1024;  // MoE matrices whose pointers and scales are staged in shared memory

struct Params {
    const uint8_t *w;           // plain GEMV: the matrix; MoE: unused
    const void *const *w_ptrs;  // MoE: device table, index = matrix; plain: null
    const float *scales;        // MoE: per-matrix scale; plain: null
    const float *x;             // [tokens][k]
    float *dst;                 // plain: [n][m]; MoE: [matrices][rows]
    int64_t k, rb;
    int rows_per_mat;           // plain: m; MoE: n_ff
    int mats;                   // plain: 1; MoE: 2 * n_pairs
    int n_pairs, n_used, tokens;
    int rpw, wpr, rt;           // rows per warp / warps per row / rows per stage
    int stages_per_mat, total_stages;
    int stage_bytes, ring;
    int x_smem_bytes;           // 0: X read from global memory
    uint32_t *status;
    uint64_t limit_ns;
};

struct Ctl {
    uint64_t full[MAX_RING], empty[MAX_RING], xbar;
    const uint8_t *mptr[MAX_TABLE];  // MoE matrix pointers (when mats <= MAX_TABLE)
    float mscale[MAX_TABLE];
    int bad[MAX_RING];
    int abort;
    int pad;
};
}  // namespace gv

// Wait with no early exit on abort, for copies already in flight.
__device__ __forceinline__ bool mbar_wait_drain_any(uint64_t *bar, uint32_t parity, uint32_t *status,
                                                    uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Group decoders for the dot products: 8 weights of one scale region as small
// exact values v[j] plus the region's scale, so that
//     sum_j W_j x_j = scale * sum_j v_j x_j            (Q4_0, Q8_0, Q6_K, NVFP4)
//     sum_j W_j x_j = a * sum_j q_j x_j - b * sum_j x_j (Q4_K: W = a q - b)
// The integer-valued codes become floats by placing them under the exponent of
// 2^23 and subtracting 2^23 (plus the code's bias), all exact and all on the
// integer and FMA pipes (no conversion instructions).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float byte_as_float(uint32_t word, int j, float minus) {
    return __uint_as_float(__byte_perm(word, 0x4B000000u, 0x7440u | static_cast<uint32_t>(j))) - minus;
}

struct Grp {
    float v[8];
    float scale;   // multiplies sum v x
    float offset;  // Q4_K: b, subtracted as b * sum x (0 otherwise)
};

template <int F> __device__ __forceinline__ void grp8(const uint8_t *row, int64_t e0, int64_t k, Grp &g);

template <> __device__ __forceinline__ void grp8<QMM_F32>(const uint8_t *row, int64_t e0, int64_t k, Grp &g) {
    decode8_f32<LdS>(row, e0, k, g.v);
    g.scale = 1.0f;
    g.offset = 0.0f;
}

template <> __device__ __forceinline__ void grp8<QMM_Q4_0>(const uint8_t *row, int64_t e0, int64_t, Grp &g) {
    const uint8_t *blk = row + (e0 >> 5) * 18;
    const int e = static_cast<int>(e0 & 31);
    g.scale = half_bits_to_f32(LdS::u16(blk));
    g.offset = 0.0f;
    const uint8_t *q = blk + 2 + (e & 15);
    uint32_t lo = ld_u32_a2<LdS>(q), hi = ld_u32_a2<LdS>(q + 4);
    if (e >= 16) {
        lo >>= 4;
        hi >>= 4;
    }
    lo &= 0x0F0F0F0Fu;
    hi &= 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g.v[j] = byte_as_float(lo, j, 8388616.0f);  // q - 8
        g.v[4 + j] = byte_as_float(hi, j, 8388616.0f);
    }
}

template <> __device__ __forceinline__ void grp8<QMM_Q8_0>(const uint8_t *row, int64_t e0, int64_t, Grp &g) {
    const uint8_t *blk = row + (e0 >> 5) * 34;
    const int e = static_cast<int>(e0 & 31);
    g.scale = half_bits_to_f32(LdS::u16(blk));
    g.offset = 0.0f;
    const uint8_t *q = blk + 2 + e;
    const uint32_t lo = ld_u32_a2<LdS>(q) ^ 0x80808080u, hi = ld_u32_a2<LdS>(q + 4) ^ 0x80808080u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g.v[j] = byte_as_float(lo, j, 8388736.0f);  // (q + 128) - 128
        g.v[4 + j] = byte_as_float(hi, j, 8388736.0f);
    }
}

template <> __device__ __forceinline__ void grp8<QMM_Q4_K>(const uint8_t *row, int64_t e0, int64_t, Grp &g) {
    const uint8_t *blk = row + (e0 >> 8) * 144;
    const int e = static_cast<int>(e0 & 255);
    const uint32_t dd = LdS::u32(blk);
    int sc, mn;
    q4k_sc_min<LdS>(blk + 4, e >> 5, sc, mn);
    g.scale = __fmul_rn(half_bits_to_f32(dd & 0xFFFFu), static_cast<float>(sc));
    g.offset = __fmul_rn(half_bits_to_f32(dd >> 16), static_cast<float>(mn));
    const int c = e >> 6, r = e & 63;
    uint2 q = LdS::u64(blk + 16 + 32 * c + (r & 31));
    if (r >= 32) {
        q.x >>= 4;
        q.y >>= 4;
    }
    q.x &= 0x0F0F0F0Fu;
    q.y &= 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g.v[j] = byte_as_float(q.x, j, 8388608.0f);
        g.v[4 + j] = byte_as_float(q.y, j, 8388608.0f);
    }
}

template <> __device__ __forceinline__ void grp8<QMM_Q6_K>(const uint8_t *row, int64_t e0, int64_t, Grp &g) {
    const uint8_t *blk = row + (e0 >> 8) * 210;
    const int e = static_cast<int>(e0 & 255);
    const int h = e >> 7, rr = e & 127, s = rr >> 5, l = rr & 31;
    const float d = half_bits_to_f32(LdS::u16(blk + 208));
    g.scale = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(LdS::u8(blk + 192 + 8 * h + (l >> 4) + 2 * s))));
    g.offset = 0.0f;
    const uint8_t *ql = blk + 64 * h + l + 32 * (s & 1);
    const uint8_t *qh = blk + 128 + 32 * h + l;
    const int lsh = (s >= 2) ? 4 : 0, hsh = 2 * s;
    const uint32_t q0 = ((ld_u32_a2<LdS>(ql) >> lsh) & 0x0F0F0F0Fu) | (((ld_u32_a2<LdS>(qh) >> hsh) & 0x03030303u) << 4);
    const uint32_t q1 =
        ((ld_u32_a2<LdS>(ql + 4) >> lsh) & 0x0F0F0F0Fu) | (((ld_u32_a2<LdS>(qh + 4) >> hsh) & 0x03030303u) << 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g.v[j] = byte_as_float(q0, j, 8388640.0f);  // q - 32
        g.v[4 + j] = byte_as_float(q1, j, 8388640.0f);
    }
}

// Four E2M1 codes (the low 16 bits of `sel`, one per nibble) -> four bytes
// 2*value + 12 (0..24), by byte permutation only.  The positive table covers
// codes 0..7; a code with its sign bit set makes the permute replicate the
// (clear) top bit of its table byte, giving 0.  The negative table is indexed
// with the sign bits flipped, so for every code one of the two lookups is 0
// and the OR is the other.
// (PTX prmt in its default mode: a selector nibble's top bit asks for the
// sign of the chosen byte replicated; __byte_perm ignores that bit.)
__device__ __forceinline__ uint32_t prmt_signed(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t e2m1x4_offset_bytes(uint32_t sel) {
    const uint32_t pos = prmt_signed(0x0F0E0D0Cu, 0x18141210u, sel);           // 12 + 2*{0,.5,1,1.5,2,3,4,6}
    const uint32_t neg = prmt_signed(0x090A0B0Cu, 0x00040608u, sel ^ 0x8888u);  // 12 - 2*{0,.5,1,1.5,2,3,4,6}
    return pos | neg;
}

template <> __device__ __forceinline__ void grp8<QMM_NVFP4>(const uint8_t *row, int64_t e0, int64_t, Grp &g) {
    const uint8_t *blk = row + (e0 >> 6) * 36;
    const int e = static_cast<int>(e0 & 63);
    g.scale = 0.5f * e4m3_to_f32(LdS::u8(blk + (e >> 4)));  // the bytes below hold 2 * value
    g.offset = 0.0f;
    const uint32_t codes = LdS::u32(blk + 4 + (e >> 1));
    const uint32_t lo = e2m1x4_offset_bytes(codes & 0xFFFFu), hi = e2m1x4_offset_bytes(codes >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g.v[j] = byte_as_float(lo, j, 8388620.0f);  // (2v + 12) - 12
        g.v[4 + j] = byte_as_float(hi, j, 8388620.0f);
    }
}

// 8 consecutive X values of one activation row (shared or global memory).
__device__ __forceinline__ void load_x8(const float *xr, bool in_smem, int64_t e0, int64_t k, float (&v)[8]) {
    if (e0 + 8 <= k && (k % 4) == 0) {
        float4 a, b;
        if (in_smem) {
            a = *reinterpret_cast<const float4 *>(xr + e0);
            b = *reinterpret_cast<const float4 *>(xr + e0 + 4);
        } else {
            a = __ldg(reinterpret_cast<const float4 *>(xr + e0));
            b = __ldg(reinterpret_cast<const float4 *>(xr + e0) + 1);
        }
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (e0 + j < k) ? (in_smem ? xr[e0 + j] : __ldg(xr + e0 + j)) : 0.0f;
    }
}

__device__ __forceinline__ void named_sync_compute() {
    asm volatile("bar.sync 1, %0;" ::"r"(32 * gv::COMPUTE_WARPS) : "memory");
}

// Two CTAs per SM for n <= 2 (more warps to hide latency), one otherwise.
template <int NV> constexpr int gemv_ctas_per_sm() { return NV <= 2 ? 2 : 1; }

template <int F, int NV>
__global__ void __launch_bounds__(gv::THREADS, gemv_ctas_per_sm<NV>()) gemv_kernel(const gv::Params p) {
    using namespace gv;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    float *sX = reinterpret_cast<float *>(base);
    uint8_t *ring = base + p.x_smem_bytes;
    float *partial = reinterpret_cast<float *>(ring + p.ring * p.stage_bytes);  // [2][8 warps][NV]
    Ctl *ctl = reinterpret_cast<Ctl *>(partial + 2 * COMPUTE_WARPS * NV + (NV & 1) * 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_RING; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], COMPUTE_WARPS);
            ctl->bad[s] = 0;
        }
        mbar_init(&ctl->xbar, 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch();
    volatile int *abort = &ctl->abort;
    const bool moe = p.w_ptrs != nullptr;
    // this CTA's stages: a contiguous run, so its rows stream sequentially
    const int s_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.total_stages / gridDim.x);
    const int s_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.total_stages / gridDim.x);
    const bool table = moe && p.mats <= MAX_TABLE;
    if (table) {
        for (int i = threadIdx.x; i < p.mats; i += THREADS) {
            ctl->mptr[i] = static_cast<const uint8_t *>(p.w_ptrs[i]);
            ctl->mscale[i] = __ldg(p.scales + i);
        }
    }
    __syncthreads();

    if (warp == COMPUTE_WARPS) {
        // ---------------- producer ----------------
        if (lane == 0) {
            if (p.x_smem_bytes) {
                const uint32_t xb = static_cast<uint32_t>(p.tokens * p.k * 4);
                mbar_arrive_expect_tx(&ctl->xbar, xb);
                bulk_load_1d(sX, p.x, xb, &ctl->xbar);
            }
            int last[MAX_RING];
            for (int r = 0; r < MAX_RING; ++r) last[r] = -1;
            for (int j = 0;; ++j) {
                const int s = s_begin + j;
                if (s >= s_end) break;
                const int slot = j % p.ring;
                if (!mbar_wait_bounded(&ctl->empty[slot], ((j / p.ring) & 1) ^ 1, abort, p.status, p.limit_ns)) break;
                const int mat = s / p.stages_per_mat;
                const int r0 = (s % p.stages_per_mat) * p.rt;
                const int rows = min(p.rt, p.rows_per_mat - r0);
                const uint8_t *mp = !moe ? p.w : (table ? ctl->mptr[mat] : static_cast<const uint8_t *>(p.w_ptrs[mat]));
                if (mp == nullptr || (reinterpret_cast<uintptr_t>(mp) & 15u) != 0) {
                    ctl->bad[slot] = 1;
                    mbar_arrive(&ctl->full[slot]);
                    continue;
                }
                ctl->bad[slot] = 0;
                const uint8_t *src = mp + static_cast<int64_t>(r0) * p.rb;
                const uintptr_t a = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
                const uint32_t len = (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) - a) +
                                      static_cast<uint32_t>(rows * p.rb) + 15u) & ~15u;
                mbar_arrive_expect_tx(&ctl->full[slot], len);
                bulk_load_1d(ring + slot * p.stage_bytes, reinterpret_cast<const void *>(a), len, &ctl->full[slot]);
                last[slot] = j;
            }
            if (*abort) {
                for (int r = 0; r < p.ring; ++r)
                    if (last[r] >= 0) mbar_wait_drain_any(&ctl->full[r], (last[r] / p.ring) & 1, p.status, p.limit_ns);
                if (p.x_smem_bytes) mbar_wait_drain_any(&ctl->xbar, 0, p.status, p.limit_ns);
            }
        }
        __syncwarp();
    } else {
        // ---------------- compute warps ----------------
        // Every compute warp walks the same stage list (the warps-per-row mode
        // meets at a named barrier each stage); a wait that gives up only
        // marks the warp dead, so no warp can strand the others.
        bool dead = false;
        if (p.x_smem_bytes) dead = !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&ctl->xbar, 0, abort, p.status, p.limit_ns));
        const int64_t ngroups = (p.k + 7) / 8;
        const bool xs = p.x_smem_bytes != 0;
        for (int j = 0;; ++j) {
            const int s = s_begin + j;
            if (s >= s_end) break;
            const int slot = j % p.ring;
            const bool got = dead ? false : mbar_wait_bounded(&ctl->full[slot], (j / p.ring) & 1, abort, p.status, p.limit_ns);
            if (!__all_sync(0xFFFFFFFFu, got)) dead = true;
            const int mat = s / p.stages_per_mat;
            const int r0 = (s % p.stages_per_mat) * p.rt;
            const int rows = min(p.rt, p.rows_per_mat - r0);
            const int tok = moe ? (mat % p.n_pairs) / p.n_used : 0;
            const float *xbase = (xs ? sX : p.x) + static_cast<int64_t>(tok) * p.k;
            const float scale = !moe ? 1.0f : (table ? ctl->mscale[mat] : __ldg(p.scales + mat));
            const bool bad = !dead && ctl->bad[slot] != 0;
            const uint8_t *mp = !moe ? p.w : (table ? ctl->mptr[mat] : static_cast<const uint8_t *>(p.w_ptrs[mat]));
            const uint8_t *buf = ring + slot * p.stage_bytes +
                                 ((reinterpret_cast<uintptr_t>(mp) + static_cast<int64_t>(r0) * p.rb) & 15u);
            float acc[MAX_RPW][NV];
#pragma unroll
            for (int i = 0; i < MAX_RPW; ++i)
#pragma unroll
                for (int v = 0; v < NV; ++v) acc[i][v] = 0.0f;
            int row_first, gstart, gstep;
            if (p.wpr == 1) {
                row_first = warp * p.rpw;
                gstart = lane;
                gstep = 32;
            } else {
                row_first = warp / p.wpr;
                gstart = (warp % p.wpr) * 32 + lane;
                gstep = 32 * p.wpr;
            }
            if (!bad && !dead) {
#pragma unroll 2
                for (int64_t gi = gstart; gi < ngroups; gi += gstep) {
                    const int64_t e0 = gi * 8;
                    float xv[NV][8];
                    float xsum[NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        load_x8(xbase + static_cast<int64_t>(v) * p.k, xs, e0, p.k, xv[v]);
                        if constexpr (F == QMM_Q4_K) {
                            xsum[v] = ((xv[v][0] + xv[v][1]) + (xv[v][2] + xv[v][3])) +
                                      ((xv[v][4] + xv[v][5]) + (xv[v][6] + xv[v][7]));
                        }
                    }
#pragma unroll
                    for (int i = 0; i < MAX_RPW; ++i) {
                        const int rl = row_first + i;
                        if (i < p.rpw && rl < rows) {
                            Grp g;
                            grp8<F>(buf + static_cast<int64_t>(rl) * p.rb, e0, p.k, g);
#pragma unroll
                            for (int v = 0; v < NV; ++v) {
                                // two independent 4-term chains
                                float pa = g.v[0] * xv[v][0], pb = g.v[4] * xv[v][4];
#pragma unroll
                                for (int t = 1; t < 4; ++t) {
                                    pa = __fmaf_rn(g.v[t], xv[v][t], pa);
                                    pb = __fmaf_rn(g.v[4 + t], xv[v][4 + t], pb);
                                }
                                const float part = pa + pb;
                                if constexpr (F == QMM_Q4_K)
                                    acc[i][v] = __fmaf_rn(g.scale, part, __fmaf_rn(-g.offset, xsum[v], acc[i][v]));
                                else
                                    acc[i][v] = __fmaf_rn(g.scale, part, acc[i][v]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < MAX_RPW; ++i) {
                if (i < p.rpw) {  // uniform across the warp
#pragma unroll
                    for (int v = 0; v < NV; ++v)
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) acc[i][v] += __shfl_xor_sync(0xFFFFFFFFu, acc[i][v], o);
                }
            }
            const float nan = __int_as_float(0x7FC00000);
            if (p.wpr == 1) {
                if (lane == 0 && !dead) {
#pragma unroll
                    for (int i = 0; i < MAX_RPW; ++i) {
                        const int rl = row_first + i;
                        if (i < p.rpw && rl < rows) {
#pragma unroll
                            for (int v = 0; v < NV; ++v) {
                                const float val = bad ? nan : scale * acc[i][v];
                                if (moe)
                                    p.dst[static_cast<int64_t>(mat) * p.rows_per_mat + r0 + rl] = val;
                                else
                                    p.dst[static_cast<int64_t>(v) * p.rows_per_mat + r0 + rl] = val;
                            }
                        }
                    }
                }
            } else {
                float *pb = partial + (j & 1) * COMPUTE_WARPS * NV;
                if (lane == 0) {
#pragma unroll
                    for (int v = 0; v < NV; ++v) pb[warp * NV + v] = acc[0][v];
                }
                named_sync_compute();
                if (!dead && warp % p.wpr == 0 && lane < NV && row_first < rows) {
                    float sum = pb[warp * NV + lane];
                    for (int t = 1; t < p.wpr; ++t) sum += pb[(warp + t) * NV + lane];
                    const float val = bad ? nan : scale * sum;
                    if (moe)
                        p.dst[static_cast<int64_t>(mat) * p.rows_per_mat + r0 + row_first] = val;
                    else
                        p.dst[static_cast<int64_t>(lane) * p.rows_per_mat + r0 + row_first] = val;
                }
            }
            if (bad && threadIdx.x == 0) atomicOr(p.status, kDevBadPtr);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->empty[slot]);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static int pow2_floor(int v) {
    int r = 1;
    while (r * 2 <= v) r *= 2;
    return r;
}

// Stage geometry for rows of rb bytes: about 40 KB per stage; shared memory
// budget per CTA `budget`.
static void plan_stages(gv::Params &p, int64_t x_bytes_total, int budget) {
    using namespace gv;
    const int rows_fit = static_cast<int>(std::min<int64_t>(1 << 20, 40960 / (p.rb > 0 ? p.rb : 1)));
    if (rows_fit >= COMPUTE_WARPS) {
        p.wpr = 1;
        p.rpw = std::min(MAX_RPW, pow2_floor(rows_fit / COMPUTE_WARPS));
        p.rt = COMPUTE_WARPS * p.rpw;
    } else {
        p.rpw = 1;
        p.rt = std::max(1, pow2_floor(rows_fit));
        p.wpr = COMPUTE_WARPS / p.rt;
    }
    p.stages_per_mat = (p.rows_per_mat + p.rt - 1) / p.rt;
    p.total_stages = p.stages_per_mat * p.mats;
    p.stage_bytes = static_cast<int>(((static_cast<int64_t>(p.rt) * p.rb + 15 + 15) / 16) * 16);
    p.x_smem_bytes = 0;
    if (x_bytes_total > 0 && x_bytes_total <= budget - 2 * p.stage_bytes - 16384 && p.k % 4 == 0)
        p.x_smem_bytes = static_cast<int>((x_bytes_total + 127) / 128 * 128);
    const int ring_budget = budget - p.x_smem_bytes - static_cast<int>(sizeof(Ctl)) - 1024;
    p.ring = std::max(2, std::min(MAX_RING, ring_budget / p.stage_bytes));
}

template <int F, int NV>
static cudaError_t launch_gemv_nv(const gv::Params &p, int num_sms, cudaStream_t st) {
    using namespace gv;
    const size_t smem = 128 + static_cast<size_t>(p.x_smem_bytes) + static_cast<size_t>(p.ring) * p.stage_bytes +
                        (2 * COMPUTE_WARPS * NV + 2) * sizeof(float) + sizeof(Ctl) + 16;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<F, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int grid = std::min(p.total_stages, num_sms * gemv_ctas_per_sm<NV>());
    return launch_pdl(gemv_kernel<F, NV>, dim3(grid), dim3(THREADS), smem, st, dim3(1, 1, 1), p);
}

template <int F>
static cudaError_t launch_gemv_f(const gv::Params &p, int n, int num_sms, cudaStream_t st) {
    switch (n) {
    case 1: return launch_gemv_nv<F, 1>(p, num_sms, st);
    case 2: return launch_gemv_nv<F, 2>(p, num_sms, st);
    case 3: return launch_gemv_nv<F, 3>(p, num_sms, st);
    case 4: return launch_gemv_nv<F, 4>(p, num_sms, st);
    case 5: return launch_gemv_nv<F, 5>(p, num_sms, st);
    case 6: return launch_gemv_nv<F, 6>(p, num_sms, st);
    case 7: return launch_gemv_nv<F, 7>(p, num_sms, st);
    case 8: return launch_gemv_nv<F, 8>(p, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

static cudaError_t dispatch(int dtype, const gv::Params &p, int n, int num_sms, cudaStream_t st) {
    switch (dtype) {
    case QMM_F32: return launch_gemv_f<QMM_F32>(p, n, num_sms, st);
    case QMM_Q4_0: return launch_gemv_f<QMM_Q4_0>(p, n, num_sms, st);
    case QMM_Q8_0: return launch_gemv_f<QMM_Q8_0>(p, n, num_sms, st);
    case QMM_Q4_K: return launch_gemv_f<QMM_Q4_K>(p, n, num_sms, st);
    case QMM_Q6_K: return launch_gemv_f<QMM_Q6_K>(p, n, num_sms, st);
    case QMM_NVFP4: return launch_gemv_f<QMM_NVFP4>(p, n, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(int dtype, const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k, int n,
                        int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    gv::Params p = {};
    p.w = static_cast<const uint8_t *>(w);
    p.x = x;
    p.dst = dst;
    p.k = k;
    p.rb = rb;
    p.rows_per_mat = static_cast<int>(m);
    p.mats = 1;
    p.n_pairs = 1;
    p.n_used = 1;
    p.tokens = n;
    p.status = status;
    p.limit_ns = limit_ns;
    plan_stages(p, static_cast<int64_t>(n) * k * 4, n <= 2 ? gv::SMEM_BUDGET / 2 : gv::SMEM_BUDGET);
    return dispatch(dtype, p, n, num_sms, st);
}

cudaError_t launch_moe_gemv(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const float *x,
                            float *y, int64_t in_f, int64_t n_ff, int n_used, int n_pairs, int tokens, int num_sms,
                            uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    gv::Params p = {};
    p.w_ptrs = w_ptrs;
    p.scales = scales;
    p.x = x;
    p.dst = y;
    p.k = in_f;
    p.rb = rb;
    p.rows_per_mat = static_cast<int>(n_ff);
    p.mats = 2 * n_pairs;
    p.n_pairs = n_pairs;
    p.n_used = n_used;
    p.tokens = tokens;
    p.status = status;
    p.limit_ns = limit_ns;
    plan_stages(p, static_cast<int64_t>(tokens) * in_f * 4, gv::SMEM_BUDGET / 2);
    return dispatch(dtype, p, 1, num_sms, st);
}

}  // namespace qmm
