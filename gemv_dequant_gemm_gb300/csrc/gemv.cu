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
// The MoE down projection runs the same kernel with one matrix per (token,
// expert) pair, each pair multiplying its own activation row, and a small
// combine kernel sums each token's pairs in a fixed order.
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
#include "l2hint.cuh"
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

// Warm L2 with this CTA's share of a plain GEMV's weights (its contiguous
// stages) before waiting for the kernel in front, so the weight stream that
// starts after the wait reads from L2.
__device__ __forceinline__ void prefetch_own_rows_l2(const uint8_t *w, int64_t rb, int64_t rows, int64_t r0,
                                                     int64_t r1) {
    if (r1 > rows) r1 = rows;
    if (r0 >= r1) return;
    const uintptr_t base = reinterpret_cast<uintptr_t>(w);
    prefetch_l2_range(base + static_cast<uintptr_t>(r0 * rb), base + static_cast<uintptr_t>(r1 * rb));
}

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
        if (p.w_ptrs == nullptr)
            prefetch_own_rows_l2(p.w, p.rb, p.rows_per_mat,
                                 static_cast<int64_t>(blockIdx.x) * p.total_stages / gridDim.x * p.rt,
                                 static_cast<int64_t>(blockIdx.x + 1) * p.total_stages / gridDim.x * p.rt);
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
// Register-X GEMV: for small n the X values each thread needs stay in its
// registers for the whole launch, so per weight only the packed bytes are read
// from shared memory.  A thread owns fixed k slices ("units" of UW weights,
// one scale region of NVFP4 or 8 weights otherwise): unit u = tk + TK*j of
// every row, j < J, where tk is the thread's index in its k team of TK
// threads.  The 256 compute threads form 256/TK teams; a stage holds
// teams*RT rows, team t taking rows t*RT .. t*RT+RT-1.  Rows are handled in
// groups of four: each warp reduces the group's 4*NVP sums (NVP = n rounded
// up to a power of two) across its lanes with a butterfly that leaves value
// i in lane i, and writes them to a per-warp partial buffer.  The producer
// warp, when the stage's slot comes back to it, adds the partials of a
// team's warps in warp order and stores the results.
// Grouped mode (the MoE down projection): a stage holds the same rows of
// all `group` pair matrices of one token, one slice per matrix, and team u
// takes every row of pair u's slice with that pair's activation row in its
// registers; the producer then sums the pairs of each row in pair order into
// dst [tokens][rows], so no workspace and no second kernel are needed.
// ---------------------------------------------------------------------------
namespace gr {
constexpr int COMPUTE_WARPS = 16;
constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);
constexpr int NT = 32 * COMPUTE_WARPS;  // compute threads
constexpr int MAX_RING = 8;
constexpr int XREG = 32;                // X floats one thread holds
constexpr int PART = 32;                // partial sums per warp and stage
constexpr int MAX_TABLE = 256;
constexpr int SMEM_BUDGET = 226 * 1024;

struct Params {
    const uint8_t *w;
    const void *const *w_ptrs;
    const float *scales;
    const float *x;
    float *dst;
    int64_t k, rb;
    int rows_per_mat, mats, n_pairs, n_used, tokens;
    int tk, J, rt, teams, stage_rows;
    int stages_per_mat, total_stages, stage_bytes, ring;
    int group;      // grouped mode: pairs per token (0: off); stages then walk (token, row block)
    int sub_bytes;  // grouped mode: bytes of one matrix's slice of a stage
    uint32_t *status;
    uint64_t limit_ns;
};

struct Ctl {
    uint64_t full[MAX_RING], empty[MAX_RING];
    const uint8_t *mptr[MAX_TABLE];
    float mscale[MAX_TABLE];
    int bad[MAX_RING];
    int abort;
    int pad;
};

template <int F> constexpr bool is_fp4() { return F == QMM_NVFP4 || F == QMM_NVFP4_V2; }
template <int F> struct Unit { static constexpr int W = is_fp4<F>() ? 16 : 8; };
template <int NV> constexpr int nv_pow2() { return NV <= 1 ? 1 : (NV <= 2 ? 2 : (NV <= 4 ? 4 : 8)); }
template <int F, int NV> constexpr int jmax() {
    return XREG / (NV * Unit<F>::W) >= 1 ? XREG / (NV * Unit<F>::W) : 1;
}
}  // namespace gr

// Units of UW weights: values v (exact small numbers), scale, Q4_K offset.
template <int F, int UW> struct UnitDec;
template <int F> struct UnitDec<F, 8> {
    static __device__ __forceinline__ void run(const uint8_t *row, int64_t e0, int64_t k, float (&v)[8], float &scale,
                                               float &offset) {
        Grp g;
        grp8<F>(row, e0, k, g);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = g.v[j];
        scale = g.scale;
        offset = g.offset;
    }
};
// NVFP4: 16 weights of one scale region (e0 % 16 == 0): v = 2 * e2m1 value,
// scale = e4m3 / 2.
template <> struct UnitDec<QMM_NVFP4, 16> {
    static __device__ __forceinline__ void run(const uint8_t *row, int64_t e0, int64_t, float (&v)[16], float &scale,
                                               float &offset) {
        const uint8_t *blk = row + (e0 >> 6) * 36;
        const int e = static_cast<int>(e0 & 63);
        scale = 0.5f * e4m3_to_f32(LdS::u8(blk + (e >> 4)));
        offset = 0.0f;
        const uint32_t c0 = LdS::u32(blk + 4 + (e >> 1)), c1 = LdS::u32(blk + 8 + (e >> 1));
        const uint32_t b[4] = {e2m1x4_offset_bytes(c0), e2m1x4_offset_bytes(c0 >> 16), e2m1x4_offset_bytes(c1),
                               e2m1x4_offset_bytes(c1 >> 16)};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) v[4 * q + j] = byte_as_float(b[q], j, 8388620.0f);
    }
};

// 16 NVFP4 weights of one scale region (codes at shared address `codes`,
// scale byte at `scb`) as 8 exact f32 pairs of their E2M1 values; *scale
// receives the e4m3 scale.
__device__ __forceinline__ void nvfp4_unit16(uint32_t codes, uint32_t scb, uint64_t (&w2)[8], float &scale) {
    const uint32_t c0 = lds32(codes), c1 = lds32(codes + 4);
    scale = e4m3_to_f32(lds8(scb));
    e2m1x8_to_f2(c0, w2);
    e2m1x8_to_f2(c1, w2 + 4);
}

// sum_i w2[i] . x2[i] over 8 pairs, two f32x2 chains.
__device__ __forceinline__ float dot16_f2(const uint64_t (&w2)[8], const uint64_t (&x2)[8]) {
    uint64_t a0 = f2_fma(w2[0], x2[0], f2_pack(0.0f, 0.0f));
    uint64_t a1 = f2_fma(w2[1], x2[1], f2_pack(0.0f, 0.0f));
#pragma unroll
    for (int q = 1; q < 4; ++q) {
        a0 = f2_fma(w2[2 * q], x2[2 * q], a0);
        a1 = f2_fma(w2[2 * q + 1], x2[2 * q + 1], a1);
    }
    const float2 s0 = f2_unpack(a0), s1 = f2_unpack(a1);
    return (s0.x + s0.y) + (s1.x + s1.y);
}

// UW consecutive X values of one activation row (zero past k).
template <int UW> __device__ __forceinline__ void load_xu(const float *xr, int64_t e0, int64_t k, float (&v)[UW]) {
    if (e0 + UW <= k && (k % 4) == 0) {
#pragma unroll
        for (int q = 0; q < UW / 4; ++q) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(xr + e0) + q);
            v[4 * q] = a.x;
            v[4 * q + 1] = a.y;
            v[4 * q + 2] = a.z;
            v[4 * q + 3] = a.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < UW; ++j) v[j] = (e0 + j < k) ? __ldg(xr + e0 + j) : 0.0f;
    }
}

// Position of a CTA's current stage in its contiguous run of stages: matrix,
// stage within the matrix, ring slot and ring phase, advanced stage by stage
// without divisions.
struct StageWalk {
    int mat, sp, slot;
    uint32_t ph;
    __device__ __forceinline__ StageWalk(int s, int stages_per_mat)
        : mat(s / stages_per_mat), sp(s - (s / stages_per_mat) * stages_per_mat), slot(0), ph(0) {}
    __device__ __forceinline__ void next(int stages_per_mat, int ring) {
        if (++sp == stages_per_mat) {
            sp = 0;
            ++mat;
        }
        if (++slot == ring) {
            slot = 0;
            ph ^= 1u;
        }
    }
};

// Grouped mode, one row: the 16 warps' partials (team u = warps u*WPT ..),
// each team's summed in warp order and scaled by sc[u], the teams added in
// order.  All loads first (compile-time indices), then the arithmetic.
template <int WPT> __device__ __forceinline__ float group_row_sum(const float *pb, int o, const float *sc) {
    constexpr int W = gr::COMPUTE_WARPS, G = W / WPT;
    float v[W], s[G];
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = pb[i * gr::PART + o];
#pragma unroll
    for (int u = 0; u < G; ++u) s[u] = sc[u];
    float a = 0.0f;
#pragma unroll
    for (int u = 0; u < G; ++u) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < WPT; ++w) sum += v[u * WPT + w];
        const float t = s[u] * sum;
        a = u == 0 ? t : a + t;
    }
    return a;
}

template <int F, int NV, int JM>
__global__ void __launch_bounds__(gr::THREADS, 1) gemv_rx_kernel(const gr::Params p) {
    using namespace gr;
    constexpr int UW = Unit<F>::W;
    constexpr int NVP = nv_pow2<NV>();
    constexpr int RG = 4;            // rows per group
    constexpr int V = RG * NVP;      // values reduced per group
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    float *partial = reinterpret_cast<float *>(ring + p.ring * p.stage_bytes);  // [ring][8 warps][PART]
    Ctl *ctl = reinterpret_cast<Ctl *>(partial + p.ring * COMPUTE_WARPS * PART);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_RING; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], COMPUTE_WARPS);
            ctl->bad[s] = 0;
        }
        ctl->abort = 0;
        fence_barrier_init();
        if (p.w_ptrs == nullptr)
            prefetch_own_rows_l2(p.w, p.rb, p.rows_per_mat,
                                 static_cast<int64_t>(blockIdx.x) * p.total_stages / gridDim.x * p.stage_rows,
                                 static_cast<int64_t>(blockIdx.x + 1) * p.total_stages / gridDim.x * p.stage_rows);
    }
    __syncthreads();
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch();
    volatile int *abort = &ctl->abort;
    const bool moe = p.w_ptrs != nullptr;
    const int s_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.total_stages / gridDim.x);
    const int s_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.total_stages / gridDim.x);
    const int nst = s_end - s_begin;
    const bool table = moe && p.mats <= MAX_TABLE;
    if (table) {
        for (int i = threadIdx.x; i < p.mats; i += THREADS) {
            ctl->mptr[i] = static_cast<const uint8_t *>(p.w_ptrs[i]);
            ctl->mscale[i] = __ldg(p.scales + i);
        }
    }
    __syncthreads();
    const float nan = __int_as_float(0x7FC00000);

    if (warp == COMPUTE_WARPS) {
        // ---------------- producer: stage loads and the cross-warp sums ----------------
        const int wpt = p.tk / 32;  // warps per team
        int issued = 0;
        StageWalk ld(s_begin, p.stages_per_mat), sw(s_begin, p.stages_per_mat);  // loads; sums (ring behind)
        for (int j = 0; j < nst + p.ring; ++j) {
            const int slot = ld.slot;  // = j % ring, for the stage loaded and the one summed
            if (j >= p.ring) {
                // the stage that used this slot, jr = j - ring, has been consumed by every compute warp
                {
                    const bool ok = mbar_wait_bounded(&ctl->empty[slot], sw.ph, abort, p.status, p.limit_ns);
                    if (!__all_sync(0xFFFFFFFFu, ok)) break;
                    const int mat = sw.mat;
                    const int r0 = sw.sp * p.stage_rows;
                    const int rows = min(p.stage_rows, p.rows_per_mat - r0);
                    const bool bad = ctl->bad[slot] != 0;
                    const float *pb = partial + slot * COMPUTE_WARPS * PART;
                    if (p.group) {
                        // token `mat`: each pair's row sum scaled, then the pairs
                        // added in pair order (NV == 1)
                        const float *sc = table ? ctl->mscale + mat * p.group : p.scales + mat * p.group;
                        for (int o = lane; o < rows; o += 32) {
                            float a;
                            switch (wpt) {
                            case 1: a = group_row_sum<1>(pb, o, sc); break;
                            case 2: a = group_row_sum<2>(pb, o, sc); break;
                            case 4: a = group_row_sum<4>(pb, o, sc); break;
                            case 8: a = group_row_sum<8>(pb, o, sc); break;
                            default: a = group_row_sum<16>(pb, o, sc); break;
                            }
                            p.dst[static_cast<int64_t>(mat) * p.rows_per_mat + r0 + o] = bad ? nan : a;
                        }
                    } else {
                        const float scale = !moe ? 1.0f : (table ? ctl->mscale[mat] : __ldg(p.scales + mat));
                        for (int o = lane; o < rows * NV; o += 32) {
                            const int rl = o / NV, v = o % NV;
                            const int tm = rl / p.rt, i = rl % p.rt;
                            float sum = 0.0f;
                            for (int w = 0; w < wpt; ++w) sum += pb[(tm * wpt + w) * PART + i * NVP + v];
                            const float val = bad ? nan : scale * sum;
                            if (moe)
                                p.dst[static_cast<int64_t>(mat) * p.rows_per_mat + r0 + rl] = val;
                            else
                                p.dst[static_cast<int64_t>(v) * p.rows_per_mat + r0 + rl] = val;
                        }
                    }
                    if (bad && lane == 0) atomicOr(p.status, kDevBadPtr);
                }
                sw.next(p.stages_per_mat, p.ring);
            }
            if (j < nst && lane == 0 && p.group) {
                // grouped: the stage's rows of each of token `mat`'s pair
                // matrices, one bulk copy per matrix into its slice
                const int mat = ld.mat;
                const int r0 = ld.sp * p.stage_rows;
                const int rows = min(p.stage_rows, p.rows_per_mat - r0);
                bool ok = true;
                uint32_t tx = 0;
                for (int u = 0; u < p.group; ++u) {
                    const int pr = mat * p.group + u;
                    const uint8_t *mp = table ? ctl->mptr[pr] : static_cast<const uint8_t *>(p.w_ptrs[pr]);
                    if (mp == nullptr || (reinterpret_cast<uintptr_t>(mp) & 15u) != 0) ok = false;
                    const uintptr_t src = reinterpret_cast<uintptr_t>(mp) + static_cast<uintptr_t>(r0) * p.rb;
                    tx += ((static_cast<uint32_t>(src & 15u) + static_cast<uint32_t>(rows * p.rb)) + 15u) & ~15u;
                }
                ctl->bad[slot] = ok ? 0 : 1;
                if (!ok) {
                    mbar_arrive(&ctl->full[slot]);
                } else {
                    mbar_arrive_expect_tx(&ctl->full[slot], tx);
                    for (int u = 0; u < p.group; ++u) {
                        const int pr = mat * p.group + u;
                        const uint8_t *mp = table ? ctl->mptr[pr] : static_cast<const uint8_t *>(p.w_ptrs[pr]);
                        const uint8_t *src = mp + static_cast<int64_t>(r0) * p.rb;
                        const uintptr_t a = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
                        const uint32_t len = (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) - a) +
                                              static_cast<uint32_t>(rows * p.rb) + 15u) & ~15u;
                        bulk_load_1d(ring + slot * p.stage_bytes + u * p.sub_bytes, reinterpret_cast<const void *>(a),
                                     len, &ctl->full[slot]);
                    }
                }
            } else if (j < nst && lane == 0) {
                const int mat = ld.mat;
                const int r0 = ld.sp * p.stage_rows;
                const int rows = min(p.stage_rows, p.rows_per_mat - r0);
                const uint8_t *mp = !moe ? p.w : (table ? ctl->mptr[mat] : static_cast<const uint8_t *>(p.w_ptrs[mat]));
                if (mp == nullptr || (reinterpret_cast<uintptr_t>(mp) & 15u) != 0) {
                    ctl->bad[slot] = 1;
                    mbar_arrive(&ctl->full[slot]);
                } else {
                    ctl->bad[slot] = 0;
                    const uint8_t *src = mp + static_cast<int64_t>(r0) * p.rb;
                    const uintptr_t a = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
                    const uint32_t len = (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) - a) +
                                          static_cast<uint32_t>(rows * p.rb) + 15u) & ~15u;
                    mbar_arrive_expect_tx(&ctl->full[slot], len);
                    bulk_load_1d(ring + slot * p.stage_bytes, reinterpret_cast<const void *>(a), len, &ctl->full[slot]);
                }
            }
            if (j < nst) ++issued;
            ld.next(p.stages_per_mat, p.ring);
            __syncwarp();
        }
        // on abort: copies still in flight land before the CTA exits
        if (lane == 0 && *abort) {
            for (int j = max(0, issued - p.ring); j < issued; ++j)
                mbar_wait_drain_any(&ctl->full[j % p.ring], (j / p.ring) & 1, p.status, p.limit_ns);
        }
        __syncwarp();
    } else {
        // ---------------- compute warps ----------------
        const int tid = threadIdx.x;
        const int team = tid / p.tk, tk = tid % p.tk;
        float xr[JM][NV][UW];
        float xs[JM][NV];  // per-unit sums of X (Q4_K minimum term)
        uint64_t x2[JM][NV][8];  // NVFP4: X as f32 pairs
        uint32_t scoff[JM], cdoff[JM];  // NVFP4: byte offsets of each unit's scale and codes in a row
        if constexpr (F == QMM_NVFP4) {
#pragma unroll
            for (int jj = 0; jj < JM; ++jj) {
                const uint32_t e0 = static_cast<uint32_t>(tk + p.tk * jj) * 16u;
                const uint32_t blk = (e0 >> 6) * 36u, e = e0 & 63u;
                scoff[jj] = blk + (e >> 4);
                cdoff[jj] = blk + 4u + (e >> 1);
            }
        } else if constexpr (F == QMM_NVFP4_V2) {
#pragma unroll
            for (int jj = 0; jj < JM; ++jj) {
                const uint32_t e0 = static_cast<uint32_t>(tk + p.tk * jj) * 16u;
                scoff[jj] = static_cast<uint32_t>(p.k >> 1) + (e0 >> 4);
                cdoff[jj] = e0 >> 1;
            }
        }
        int cur_tok = -1, cur_mat = -1, tok = 0;
        bool dead = false;
        StageWalk wk(s_begin, p.stages_per_mat);
        for (int j = 0; j < nst; ++j, wk.next(p.stages_per_mat, p.ring)) {
            const int slot = wk.slot;
            const int mat = wk.mat;
            if (mat != cur_mat) {  // uniform over the CTA (the team's, grouped): the stage decides it
                cur_mat = mat;
                tok = p.group ? mat * p.group + team : (moe ? (mat % p.n_pairs) / p.n_used : 0);
            }
            if (tok != cur_tok) {
                cur_tok = tok;
#pragma unroll
                for (int jj = 0; jj < JM; ++jj) {
                    const int u = tk + p.tk * jj;  // every unit exists: the team covers k exactly
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        load_xu<UW>(p.x + static_cast<int64_t>(tok + v) * p.k, static_cast<int64_t>(u) * UW, p.k,
                                    xr[jj][v]);
                        float t = 0.0f;
#pragma unroll
                        for (int w = 0; w < UW; ++w) t += xr[jj][v][w];
                        xs[jj][v] = t;
                        if constexpr (is_fp4<F>()) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                x2[jj][v][q] = f2_pack(xr[jj][v][2 * q], xr[jj][v][2 * q + 1]);
                        }
                    }
                }
            }
            const bool got = dead ? false : mbar_wait_bounded(&ctl->full[slot], wk.ph, abort, p.status, p.limit_ns);
            if (!__all_sync(0xFFFFFFFFu, got)) dead = true;
            const int r0 = wk.sp * p.stage_rows;
            const int rows = min(p.stage_rows, p.rows_per_mat - r0);
            const bool bad = !dead && ctl->bad[slot] != 0;
            // grouped: the team's pair is activation row `tok`, its slice the team's
            const int wm = p.group ? tok : mat;
            const uint8_t *mp = !moe ? p.w : (table ? ctl->mptr[wm] : static_cast<const uint8_t *>(p.w_ptrs[wm]));
            const uint8_t *buf = ring + slot * p.stage_bytes + (p.group ? team * p.sub_bytes : 0) +
                                 ((reinterpret_cast<uintptr_t>(mp) + static_cast<int64_t>(r0) * p.rb) & 15u);
            float *pw = partial + (slot * COMPUTE_WARPS + warp) * PART;
            const uint32_t sbase = smem_u32(buf);
            // rows past the end of the matrix (last stage) are computed from
            // stale, in-bounds stage bytes and never stored
#pragma unroll 1
            for (int i0 = 0; i0 < p.rt; i0 += RG) {
                float acc[V];
#pragma unroll
                for (int q = 0; q < V; ++q) acc[q] = 0.0f;
                if (!bad && !dead) {
#pragma unroll
                    for (int r = 0; r < RG; ++r) {
                        const int rl = (p.group ? 0 : team * p.rt) + i0 + r;
                        const uint8_t *rowp = buf + static_cast<int64_t>(rl) * p.rb;
                        const uint32_t rbase = sbase + static_cast<uint32_t>(rl) * static_cast<uint32_t>(p.rb);
#pragma unroll
                        for (int jj = 0; jj < JM; ++jj) {
                            const int u = tk + p.tk * jj;
                            if constexpr (is_fp4<F>()) {
                                uint64_t w2[8];
                                float sc;
                                nvfp4_unit16(rbase + cdoff[jj], rbase + scoff[jj], w2, sc);
#pragma unroll
                                for (int v = 0; v < NV; ++v)
                                    acc[r * NVP + v] = __fmaf_rn(sc, dot16_f2(w2, x2[jj][v]), acc[r * NVP + v]);
                            } else {
                                float wv[UW], sc, off;
                                UnitDec<F, UW>::run(rowp, static_cast<int64_t>(u) * UW, p.k, wv, sc, off);
#pragma unroll
                                for (int v = 0; v < NV; ++v) {
                                    float c[4];
#pragma unroll
                                    for (int q = 0; q < 4; ++q) c[q] = wv[q] * xr[jj][v][q];
#pragma unroll
                                    for (int w = 4; w < UW; ++w) c[w & 3] = __fmaf_rn(wv[w], xr[jj][v][w], c[w & 3]);
                                    const float part = (c[0] + c[1]) + (c[2] + c[3]);
                                    float &a = acc[r * NVP + v];
                                    if constexpr (F == QMM_Q4_K)
                                        a = __fmaf_rn(sc, part, __fmaf_rn(-off, xs[jj][v], a));
                                    else
                                        a = __fmaf_rn(sc, part, a);
                                }
                            }
                        }
                    }
                }
                const float red = warp_transpose_sum<V>(acc, lane);
                if (lane < V) pw[i0 * NVP + lane] = red;
            }
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

// Register-X plan: k team size TK, units per thread J, rows per team and
// stage RT; false when X does not fit in registers (then the shared-memory X
// kernel runs).
template <int F, int NV> static bool plan_rx(gr::Params &p, int num_sms) {
    using namespace gr;
    constexpr int UW = Unit<F>::W;
    constexpr int JM = jmax<F, NV>();
    if (NV * UW > XREG) return false;
    // short rows: the shared-memory X kernel has the shorter start-up and wins
    if (p.k < 2048) return false;
    if (p.k % UW != 0) return false;
    const int64_t nunits = p.k / UW;
    // a team of TK threads covers k exactly with J units each (J <= JM)
    int best_tk = 0, best_j = 0;
    for (int tk = NT; tk >= 32; tk /= 2) {
        if (nunits % tk == 0 && nunits / tk <= JM) {
            best_tk = tk;
            best_j = static_cast<int>(nunits / tk);
            break;
        }
    }
    if (best_tk == 0) return false;
    p.tk = best_tk;
    p.J = best_j;
    p.teams = NT / best_tk;
    const int rt_max = PART / nv_pow2<NV>();
    const int64_t rows_total = static_cast<int64_t>(p.rows_per_mat) * p.mats;
    // rows per team: enough stages for every SM, stages of about 40 KB at most
    int64_t rt = rows_total / (static_cast<int64_t>(p.teams) * num_sms);
    rt = std::min<int64_t>(rt, 40960 / (static_cast<int64_t>(p.teams) * std::max<int64_t>(p.rb, 1)));
    rt = std::max<int64_t>(4, std::min<int64_t>(rt, rt_max)) / 4 * 4;  // whole groups of four rows
    p.rt = static_cast<int>(rt);
    p.stage_rows = p.teams * p.rt;
    p.stages_per_mat = (p.rows_per_mat + p.stage_rows - 1) / p.stage_rows;
    p.total_stages = p.stages_per_mat * p.mats;
    p.stage_bytes = static_cast<int>((static_cast<int64_t>(p.stage_rows) * p.rb + 15 + 15) / 16 * 16);
    const int fixed = static_cast<int>(sizeof(Ctl)) + 1024;
    const int per_stage = p.stage_bytes + COMPUTE_WARPS * PART * 4;
    p.ring = std::min(MAX_RING, (SMEM_BUDGET - fixed) / per_stage);
    return p.ring >= 2;
}

template <int F, int NV, int J> static cudaError_t launch_rx_j(const gr::Params &p, int num_sms, cudaStream_t st) {
    using namespace gr;
    const size_t smem = 128 + static_cast<size_t>(p.ring) * (p.stage_bytes + COMPUTE_WARPS * PART * 4) + sizeof(Ctl) + 16;
    cudaError_t e = cudaFuncSetAttribute(gemv_rx_kernel<F, NV, J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int grid = std::min(p.total_stages, num_sms);
    return launch_pdl(gemv_rx_kernel<F, NV, J>, dim3(grid), dim3(THREADS), smem, st, dim3(1, 1, 1), p);
}

template <int F, int NV> static cudaError_t launch_rx(const gr::Params &p, int num_sms, cudaStream_t st) {
    constexpr int JM = gr::jmax<F, NV>();
    switch (p.J) {
    case 1: return launch_rx_j<F, NV, 1>(p, num_sms, st);
    case 2: if constexpr (JM >= 2) return launch_rx_j<F, NV, 2>(p, num_sms, st); else return cudaErrorInvalidValue;
    case 3: if constexpr (JM >= 3) return launch_rx_j<F, NV, 3>(p, num_sms, st); else return cudaErrorInvalidValue;
    case 4: if constexpr (JM >= 4) return launch_rx_j<F, NV, 4>(p, num_sms, st); else return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

// Grouped register-X plan for the MoE down projection: the `group` pairs of
// a token are the teams (team size 512/group threads, covering k exactly
// with J <= JM units each), and every team takes all rows of a stage: about
// 40 KB of weights per stage in whole groups of four rows, at most PART (one
// partial per row and warp), fewer while that leaves SMs without a stage.
template <int F> static bool plan_rx_group(gr::Params &p, int group, int tokens, int num_sms) {
    using namespace gr;
    constexpr int UW = Unit<F>::W;
    constexpr int JM = jmax<F, 1>();
    if (UW > XREG || p.k < 2048 || p.k % UW != 0 || group < 2 || NT % group != 0) return false;
    const int tk = NT / group;
    if (tk % 32 != 0) return false;
    const int64_t nunits = p.k / UW;
    if (nunits % tk != 0 || nunits / tk > JM) return false;
    p.tk = tk;
    p.J = static_cast<int>(nunits / tk);
    p.teams = group;
    p.group = group;
    int64_t r = 40960 / (static_cast<int64_t>(group) * std::max<int64_t>(p.rb, 1));
    r = std::max<int64_t>(4, std::min<int64_t>(r, PART)) / 4 * 4;
    while (r > 4 && static_cast<int64_t>(tokens) * ((p.rows_per_mat + r - 1) / r) < num_sms) r -= 4;
    p.rt = static_cast<int>(r);
    p.stage_rows = p.rt;
    p.stages_per_mat = (p.rows_per_mat + p.stage_rows - 1) / p.stage_rows;
    p.total_stages = p.stages_per_mat * tokens;
    // a slice holds its rows plus the source's offset from 16 bytes
    p.sub_bytes = static_cast<int>((static_cast<int64_t>(p.stage_rows) * p.rb + 15 + 15) / 16 * 16);
    p.stage_bytes = group * p.sub_bytes;
    const int fixed = static_cast<int>(sizeof(Ctl)) + 1024;
    const int per_stage = p.stage_bytes + COMPUTE_WARPS * PART * 4;
    p.ring = std::min(MAX_RING, (SMEM_BUDGET - fixed) / per_stage);
    return p.ring >= 2;
}

template <int F>
static cudaError_t launch_group_f(gr::Params rp, int group, int tokens, int num_sms, cudaStream_t st, bool *used) {
    *used = plan_rx_group<F>(rp, group, tokens, num_sms);
    return *used ? launch_rx<F, 1>(rp, num_sms, st) : cudaSuccess;
}

// The grouped down projection when its plan exists (*used), else nothing.
static cudaError_t launch_group_any(int dtype, const gr::Params &rp, int group, int tokens, int num_sms,
                                    cudaStream_t st, bool *used) {
    switch (dtype) {
    case QMM_F32: return launch_group_f<QMM_F32>(rp, group, tokens, num_sms, st, used);
    case QMM_Q4_0: return launch_group_f<QMM_Q4_0>(rp, group, tokens, num_sms, st, used);
    case QMM_Q8_0: return launch_group_f<QMM_Q8_0>(rp, group, tokens, num_sms, st, used);
    case QMM_Q4_K: return launch_group_f<QMM_Q4_K>(rp, group, tokens, num_sms, st, used);
    case QMM_Q6_K: return launch_group_f<QMM_Q6_K>(rp, group, tokens, num_sms, st, used);
    case QMM_NVFP4: return launch_group_f<QMM_NVFP4>(rp, group, tokens, num_sms, st, used);
    case QMM_NVFP4_V2: return launch_group_f<QMM_NVFP4_V2>(rp, group, tokens, num_sms, st, used);
    default: *used = false; return cudaErrorInvalidValue;
    }
}

// Register-X kernel when its plan exists, else the shared-memory X kernel.
template <int F, int NV>
static cudaError_t launch_any(gr::Params rp, const gv::Params &gp, int num_sms, cudaStream_t st) {
    if constexpr (NV * gr::Unit<F>::W <= gr::XREG) {
        if (plan_rx<F, NV>(rp, num_sms)) return launch_rx<F, NV>(rp, num_sms, st);
    }
    return launch_gemv_nv<F, NV>(gp, num_sms, st);
}

template <int F>
static cudaError_t launch_any_f(const gr::Params &rp, const gv::Params &gp, int n, int num_sms, cudaStream_t st) {
    switch (n) {
    case 1: return launch_any<F, 1>(rp, gp, num_sms, st);
    case 2: return launch_any<F, 2>(rp, gp, num_sms, st);
    case 3: return launch_any<F, 3>(rp, gp, num_sms, st);
    case 4: return launch_any<F, 4>(rp, gp, num_sms, st);
    case 5: return launch_any<F, 5>(rp, gp, num_sms, st);
    case 6: return launch_any<F, 6>(rp, gp, num_sms, st);
    case 7: return launch_any<F, 7>(rp, gp, num_sms, st);
    case 8: return launch_any<F, 8>(rp, gp, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

static cudaError_t dispatch_any(int dtype, const gr::Params &rp, const gv::Params &gp, int n, int num_sms,
                                cudaStream_t st) {
    switch (dtype) {
    case QMM_F32: return launch_any_f<QMM_F32>(rp, gp, n, num_sms, st);
    case QMM_Q4_0: return launch_any_f<QMM_Q4_0>(rp, gp, n, num_sms, st);
    case QMM_Q8_0: return launch_any_f<QMM_Q8_0>(rp, gp, n, num_sms, st);
    case QMM_Q4_K: return launch_any_f<QMM_Q4_K>(rp, gp, n, num_sms, st);
    case QMM_Q6_K: return launch_any_f<QMM_Q6_K>(rp, gp, n, num_sms, st);
    case QMM_NVFP4: return launch_any_f<QMM_NVFP4>(rp, gp, n, num_sms, st);
    case QMM_NVFP4_V2: return launch_any_f<QMM_NVFP4_V2>(rp, gp, n, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

static gr::Params rx_params(const gv::Params &g) {
    gr::Params r = {};
    r.w = g.w;
    r.w_ptrs = g.w_ptrs;
    r.scales = g.scales;
    r.x = g.x;
    r.dst = g.dst;
    r.k = g.k;
    r.rb = g.rb;
    r.rows_per_mat = g.rows_per_mat;
    r.mats = g.mats;
    r.n_pairs = g.n_pairs;
    r.n_used = g.n_used;
    r.tokens = g.tokens;
    r.status = g.status;
    r.limit_ns = g.limit_ns;
    return r;
}

cudaError_t launch_gemv(int dtype, const void *w, int64_t rb, const float *x, float *dst, int64_t m, int64_t k, int n,
                        int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    // the split-K register-X kernel first (short calls: many small CTAs); if
    // it has no plan, or its launch is refused, the kernels below run
    const cudaError_t es = launch_gemv_sk(dtype, w, rb, x, dst, m, k, n, num_sms, status, limit_ns, st);
    if (es == cudaSuccess) return es;
    if (es != cudaErrorNotSupported) (void)cudaGetLastError();
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
    return dispatch_any(dtype, rx_params(p), p, n, num_sms, st);
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
    return dispatch_any(dtype, rx_params(p), p, 1, num_sms, st);
}

// MoE down projection, combine step: y[i][r] = sum over u < n_used of
// part[i*n_used + u][r], summed in the order u = 0, 1, ... (deterministic).
// Four consecutive r per thread when gin % 4 == 0 (16-byte loads and stores).
__global__ void __launch_bounds__(256) moe_combine_kernel(const float *__restrict__ part, float *__restrict__ y,
                                                          int64_t gin, int n_used, int64_t t) {
    griddep_wait();
    griddep_launch();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if ((gin & 3) == 0) {
        const int64_t g4 = gin / 4, total = t * g4;
        for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
            const int64_t i = e / g4, c = e - i * g4;
            const float4 *src = reinterpret_cast<const float4 *>(part) + i * n_used * g4 + c;
            float4 a = src[0];
            for (int u = 1; u < n_used; ++u) {
                const float4 b = src[u * g4];
                a.x += b.x;
                a.y += b.y;
                a.z += b.z;
                a.w += b.w;
            }
            reinterpret_cast<float4 *>(y)[e] = a;
        }
    } else {
        const int64_t total = t * gin;
        for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
            const int64_t i = e / gin, r = e - i * gin;
            const float *src = part + i * n_used * gin + r;
            float a = src[0];
            for (int u = 1; u < n_used; ++u) a += src[u * gin];
            y[e] = a;
        }
    }
}

cudaError_t launch_moe_down(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const float *h,
                            float *y, float *part, int64_t n_ff, int64_t gin, int n_used, int tokens, int num_sms,
                            uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    // the grouped register-X kernel when it has a plan; else the pair
    // products -- the MoE GEMV with one matrix per pair, each pair its own
    // activation row (n_used = 1 makes the activation row the pair index) --
    // then the combine kernel
    const int n_pairs = n_used * tokens;
    gv::Params p = {};
    p.w_ptrs = w_ptrs;
    p.scales = scales;
    p.x = h;
    p.dst = n_used == 1 ? y : part;
    p.k = n_ff;
    p.rb = rb;
    p.rows_per_mat = static_cast<int>(gin);
    p.mats = n_pairs;
    p.n_pairs = n_pairs;
    p.n_used = 1;
    p.tokens = n_pairs;
    p.status = status;
    p.limit_ns = limit_ns;
    if (n_used > 1) {
        // grouped: each token's pairs in one stage, summed by the kernel into y
        gr::Params rp = rx_params(p);
        rp.dst = y;
        bool used = false;
        const cudaError_t eg = launch_group_any(dtype, rp, n_used, tokens, num_sms, st, &used);
        if (used || eg != cudaSuccess) return eg;
    }
    plan_stages(p, static_cast<int64_t>(n_pairs) * n_ff * 4, gv::SMEM_BUDGET / 2);
    cudaError_t e = dispatch_any(dtype, rx_params(p), p, 1, num_sms, st);
    if (e != cudaSuccess || n_used == 1) return e;
    return launch_moe_combine(part, y, gin, n_used, tokens, num_sms, st);
}

cudaError_t launch_moe_combine(const float *part, float *y, int64_t gin, int n_used, int tokens, int num_sms,
                               cudaStream_t st) {
    const int64_t per = (gin & 3) == 0 ? gin / 4 : gin;
    const int64_t want = (tokens * per + 255) / 256;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 4LL * num_sms)));
    return launch_pdl(moe_combine_kernel, dim3(grid), dim3(256), 0, st, dim3(1, 1, 1), part, y, gin, n_used,
                      static_cast<int64_t>(tokens));
}

}  // namespace qmm
