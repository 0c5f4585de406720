// moe_q8.cu -- the NVFP4 MoE products on int8 (Q8_1) activations.
//
// memra-engine 0.128.0 moe_rows_ceiling_bench.rs serves its gate/up GEMV on
// activations quantized by quantize_q8_1 and names the PRMT/dp4a instruction
// stream as the cost it measures; neither kernel's source is printed.  The
// product here is the exact one on the quantized activation,
//     dst[mat][r] = scales[mat] * sum_c W_mat[r][c] * q[a][c] * d[a][c/32],
// with Q8_1 blocks of 32 values (d = amax/127, q = x/d rounded half away from
// zero, both decided in float32 by the quantizer below).
//
// Arithmetic.  A 16-weight region of an NVFP4 row has one E4M3 scale s, and
// lies inside one 32-value activation block (scale d).  Its contribution is
//     sum_c e2m1_c * s * q_c * d  =  (s * d / 2) * sum_c (2 e2m1_c) q_c,
// and 2*e2m1 is an integer in [-12, 12]: the inner sum is an exact int32 dot
// product of bytes.  One byte permutation per four codes turns them into the
// unsigned bytes 2*e2m1 + 12 (0..24); dp4a multiplies four of them by four
// signed activation bytes; the +12 offset is removed by starting the sum at
// -12 * (sum of the region's 16 q), precomputed once per lane.  Per region
// that leaves one float multiply (s*d) and one FMA into a float32 lane sum of
// at most 4*J terms; lanes then meet in a fixed shuffle tree, and the row
// total is scaled by scales[mat]/2.  Results are deterministic.
//
// Layout of the work: the rows of all matrices are cut into stages of 16
// rows (one per compute warp).  A producer warp moves each stage, contiguous
// in memory, into a shared-memory ring with one bulk copy; compute warp w
// takes row w of every stage of its CTA.  Lane l owns the 64-weight groups
// l, l+32, ... of the row (J of them), and keeps the matching activation
// bytes, block scales and offset terms in registers for as long as the
// activation row stays the same.  Given the float32 activation instead of
// its Q8_1 blocks, the compute warps quantize each new activation row
// together into a small shared-memory table first (the quantizer kernel's
// steps, so the same bytes), and the lanes read their groups from there.
// Every wait is bounded; a stage with a NULL or misaligned matrix pointer is
// skipped, reported, and its rows set to NaN.
#include <cuda_fp8.h>

#include <algorithm>

#include "decode.cuh"
#include "kernels.h"

namespace qmm {

namespace mq {
constexpr int COMPUTE_WARPS = 16;
constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);
constexpr int MAX_RING = 8;
constexpr int MAX_TABLE = 512;
constexpr int SMEM_BUDGET = 226 * 1024;

struct Params {
    const void *const *w_ptrs;
    const float *scales;
    const int8_t *q;  // [act rows][k]
    const float *d;   // [act rows][k/32]
    const float *x;   // [act rows][k] float32, quantized in the kernel (q, d unused) when not null
    float *dst;       // [mats][rows_per_mat]
    int64_t k, rb;
    int rows_per_mat, mats, n_pairs, n_used;
    int stages_per_mat, total_stages, stage_bytes, ring;
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
}  // namespace mq

// Wait with no early exit on abort, for copies already in flight.
__device__ __forceinline__ bool mq_wait_drain(uint64_t *bar, uint32_t parity, uint32_t *status, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Four E4M3 scale bytes -> four floats (hardware fp8x2 -> f16x2, then exact widening).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&s)[4]) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
    s[0] = a.x;
    s[1] = a.y;
    s[2] = b.x;
    s[3] = b.y;
}

// Q8_1 arithmetic shared by the quantizer kernel and the kernels that
// quantize their activation themselves: d = amax/127, the reciprocal, and a
// code, each one float32 operation, so both produce the same bytes.
__device__ __forceinline__ float q8_block_scale(float amax) { return __fdiv_rn(amax, 127.0f); }
__device__ __forceinline__ float q8_block_inv(float d) { return d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f; }
__device__ __forceinline__ int q8_code(float v, float id) { return static_cast<int>(roundf(__fmul_rn(v, id))); }

// A float32 activation row of k values (k % 64 == 0, 16-byte aligned) as
// Q8_1 into shared memory, by the CTA's NT compute threads together: codes
// [k/64][16] words (value 4i+j of a 64-value group in byte j of word i), then
// block scales [k/64][2].  Thread i takes values 8i .. 8i+7; the four threads
// of a 32-value block meet in a shuffle for its amax.  Every thread of the
// NT calls it (the shuffles need whole warps).
template <int NT>
__device__ __forceinline__ void q8_quantize_row_shared(const float *xr, int64_t k, uint32_t *tq, float *td, int ct) {
    const int n8 = static_cast<int>(k >> 3);
    for (int base = ct & ~31; base < n8; base += NT) {
        const int i = base + (ct & 31);
        const bool ok = i < n8;
        float v[8];
        if (ok) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(xr) + 2 * i);
            const float4 c = __ldg(reinterpret_cast<const float4 *>(xr) + 2 * i + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) v[t] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(v[t]));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        if (ok) {
            const float db = q8_block_scale(amax);
            const float id = q8_block_inv(db);
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                uint32_t word = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    word |= (static_cast<uint32_t>(q8_code(v[4 * w + j], id)) & 0xFFu) << (8 * j);
                tq[2 * i + w] = word;  // group i/8, words 2(i%8), 2(i%8)+1
            }
            if ((i & 3) == 0) td[i >> 2] = db;  // block i/4 = group i/8, half (i/4)%2
        }
    }
}

// Four codes against four activation bytes: the positive lookup (negative
// codes give 0) and the lookup on the sign-flipped selector (positive codes
// give 0) each feed one dp4a, which is the dp4a of their OR.
__device__ __forceinline__ int dot4(uint32_t sel, uint32_t selx, uint32_t qw, int acc) {
    const uint32_t pos = prmt_signed(0x0F0E0D0Cu, 0x18141210u, sel);   // 12 + 2*{0,.5,1,1.5,2,3,4,6}
    const uint32_t neg = prmt_signed(0x090A0B0Cu, 0x00040608u, selx);  // 12 - 2*{0,.5,1,1.5,2,3,4,6}
    return dp4a_us(neg, qw, dp4a_us(pos, qw, acc));
}

// The exact int32 sum over a 16-weight region: its two code words (eight
// codes each) against four activation words, started at the offset term.
__device__ __forceinline__ int region_dot(uint32_t c0, uint32_t c1, const uint32_t *qw, int start) {
    const uint32_t x0 = c0 ^ 0x88888888u, x1 = c1 ^ 0x88888888u;
    int v = dot4(c0, x0, qw[0], start);
    v = dot4(c0 >> 16, x0 >> 16, qw[1], v);
    v = dot4(c1, x1, qw[2], v);
    return dot4(c1 >> 16, x1 >> 16, qw[3], v);
}

template <int F, int J, int RW, bool FX>
__global__ void __launch_bounds__(mq::THREADS, 1) moe_q8_kernel(const mq::Params p) {
    using namespace mq;
    constexpr int SR = COMPUTE_WARPS * RW;  // rows per stage: warp w takes rows w*RW .. w*RW+RW-1
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    Ctl *ctl = reinterpret_cast<Ctl *>(ring + p.ring * p.stage_bytes);
    // the quantized activation row (FX): codes [k/64][16] words, then scales [k/64][2]
    uint32_t *tq = reinterpret_cast<uint32_t *>((reinterpret_cast<uintptr_t>(ctl + 1) + 15) & ~uintptr_t(15));
    float *td = reinterpret_cast<float *>(tq + 16 * (p.k >> 6));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_RING; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], COMPUTE_WARPS);
            ctl->bad[s] = 0;
        }
        ctl->abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch();
    volatile int *abort = &ctl->abort;
    const int s_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.total_stages / gridDim.x);
    const int s_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.total_stages / gridDim.x);
    const int nst = s_end - s_begin;
    const bool table = p.mats <= MAX_TABLE;
    if (table) {
        for (int i = threadIdx.x; i < p.mats; i += THREADS) {
            ctl->mptr[i] = static_cast<const uint8_t *>(p.w_ptrs[i]);
            ctl->mscale[i] = __ldg(p.scales + i);
        }
    }
    __syncthreads();
    // the CTA's stages form one contiguous run: walk (matrix, first row) and
    // (ring slot, phase) incrementally from its first stage
    const int mat0 = s_begin / p.stages_per_mat;
    const int r00 = (s_begin - mat0 * p.stages_per_mat) * SR;

    if (warp == COMPUTE_WARPS) {
        // ---------------- producer: one bulk copy per stage ----------------
        if (lane == 0) {
            int issued = 0, mat = mat0, r0 = r00, slot = 0;
            uint32_t ph = 0;
            for (int j = 0; j < nst; ++j) {
                if (j >= p.ring && !mbar_wait_bounded(&ctl->empty[slot], ph ^ 1, abort, p.status, p.limit_ns)) break;
                const int rows = min(SR, p.rows_per_mat - r0);
                const uint8_t *mp = table ? ctl->mptr[mat] : static_cast<const uint8_t *>(p.w_ptrs[mat]);
                if (mp == nullptr || (reinterpret_cast<uintptr_t>(mp) & 15u) != 0) {
                    ctl->bad[slot] = 1;
                    mbar_arrive(&ctl->full[slot]);
                } else {
                    // SR rows of rb bytes (rb a multiple of 4): the copy covers
                    // them rounded up to 16 bytes, which stays inside the
                    // matrix's allocation granule
                    ctl->bad[slot] = 0;
                    const uint32_t len = (static_cast<uint32_t>(rows * p.rb) + 15u) & ~15u;
                    mbar_arrive_expect_tx(&ctl->full[slot], len);
                    bulk_load_1d(ring + slot * p.stage_bytes, mp + static_cast<int64_t>(r0) * p.rb, len,
                                 &ctl->full[slot]);
                }
                ++issued;
                if ((r0 += SR) >= p.rows_per_mat) {
                    r0 = 0;
                    ++mat;
                }
                if (++slot == p.ring) {
                    slot = 0;
                    ph ^= 1u;
                }
            }
            if (*abort) {  // copies still in flight land before the CTA exits
                for (int j = max(0, issued - p.ring); j < issued; ++j)
                    mq_wait_drain(&ctl->full[j % p.ring], (j / p.ring) & 1, p.status, p.limit_ns);
            }
        }
        __syncwarp();
        return;
    }

    // ---------------- compute warps ----------------
    const int U = static_cast<int>(p.k >> 6);  // 64-weight groups per row
    uint32_t qv[J][16];                        // activation bytes of each group, 4 per word
    float dd[J][2];                            // the group's two activation block scales
    int corr[J][4];                            // -12 * (sum of q) per 16-weight region
    // the stage buffer is 16-byte aligned and row w starts at w * rb
    const bool v4 = (p.rb & 15) == 0;
    int cur_mat = -1, mat = mat0, r0 = r00, slot = 0;
    uint32_t ph = 0;
    bool dead = false;
    float scale = 0.0f;
    const float nan = __int_as_float(0x7FC00000);
    for (int j = 0; j < nst; ++j) {
        if (mat != cur_mat) {  // uniform over the CTA: the stage decides it
            const int act = (mat % p.n_pairs) / p.n_used;
            const int prev_act = cur_mat < 0 ? -1 : (cur_mat % p.n_pairs) / p.n_used;
            cur_mat = mat;
            scale = 0.5f * (table ? ctl->mscale[mat] : __ldg(p.scales + mat));  // codes hold 2 * e2m1
            if (act != prev_act) {
                if constexpr (FX) {
                    // every compute warp has copied the previous row's table into
                    // its registers; quantize the new row together, then read it
                    asm volatile("bar.sync 1, %0;" ::"n"(32 * COMPUTE_WARPS) : "memory");
                    q8_quantize_row_shared<32 * COMPUTE_WARPS>(p.x + static_cast<int64_t>(act) * p.k, p.k, tq, td,
                                                               threadIdx.x);
                    asm volatile("bar.sync 1, %0;" ::"n"(32 * COMPUTE_WARPS) : "memory");
                }
#pragma unroll
                for (int jj = 0; jj < J; ++jj) {
                    const int u = lane + 32 * jj;
                    if (u < U) {
                        if constexpr (FX) {
                            const uint4 *src = reinterpret_cast<const uint4 *>(tq) + 4 * u;
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const uint4 v = src[t];
                                qv[jj][4 * t] = v.x;
                                qv[jj][4 * t + 1] = v.y;
                                qv[jj][4 * t + 2] = v.z;
                                qv[jj][4 * t + 3] = v.w;
                            }
                            dd[jj][0] = td[2 * u];
                            dd[jj][1] = td[2 * u + 1];
                        } else {
                            const uint4 *src =
                                reinterpret_cast<const uint4 *>(p.q + static_cast<int64_t>(act) * p.k) + 4 * u;
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const uint4 v = __ldg(src + t);
                                qv[jj][4 * t] = v.x;
                                qv[jj][4 * t + 1] = v.y;
                                qv[jj][4 * t + 2] = v.z;
                                qv[jj][4 * t + 3] = v.w;
                            }
                            const float2 ds = __ldg(
                                reinterpret_cast<const float2 *>(p.d + static_cast<int64_t>(act) * (p.k >> 5)) + u);
                            dd[jj][0] = ds.x;
                            dd[jj][1] = ds.y;
                        }
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            int sum = 0;
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                sum = __dp4a(static_cast<int>(qv[jj][4 * r + t]), 0x01010101, sum);
                            corr[jj][r] = -12 * sum;
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) qv[jj][t] = 0u;
                        dd[jj][0] = dd[jj][1] = 0.0f;
#pragma unroll
                        for (int r = 0; r < 4; ++r) corr[jj][r] = 0;
                    }
                }
            }
        }
        const bool got = dead ? false : mbar_wait_bounded(&ctl->full[slot], ph, abort, p.status, p.limit_ns);
        if (!__all_sync(0xFFFFFFFFu, got)) dead = true;
        const int rows = min(SR, p.rows_per_mat - r0);
        const bool bad = !dead && ctl->bad[slot] != 0;
        const int row0 = warp * RW;
        if (!dead && row0 < rows) {
            float acc[RW];
#pragma unroll
            for (int rr = 0; rr < RW; ++rr) acc[rr] = 0.0f;
            if (!bad) {
                const uint32_t st0 = smem_u32(ring + slot * p.stage_bytes);
#pragma unroll
                for (int jj = 0; jj < J; ++jj) {
                    const int u = lane + 32 * jj;
                    if (u < U) {
#pragma unroll
                        for (int rr = 0; rr < RW; ++rr) {
                            // a row past the matrix's end (last stage) reads
                            // in-bounds stale stage bytes and is never stored
                            const uint32_t rowa = st0 + static_cast<uint32_t>((row0 + rr) * p.rb);
                            uint32_t cw[8], sw;
                            if constexpr (F == QMM_NVFP4) {
                                const uint32_t g = rowa + 36u * static_cast<uint32_t>(u);
                                sw = ld_shared_u32(g);
#pragma unroll
                                for (int t = 0; t < 8; ++t) cw[t] = ld_shared_u32(g + 4u + 4u * t);
                            } else {  // V2: codes at u*32, scales at k/2 + 4u
                                const uint32_t g = rowa + 32u * static_cast<uint32_t>(u);
                                if (v4) {  // rows start on 16 bytes: two 16-byte loads
                                    const uint4 a = ld_shared_v4(g), b = ld_shared_v4(g + 16u);
                                    cw[0] = a.x; cw[1] = a.y; cw[2] = a.z; cw[3] = a.w;
                                    cw[4] = b.x; cw[5] = b.y; cw[6] = b.z; cw[7] = b.w;
                                } else {  // rows start on 4 bytes only (rb = 36 * k/64)
#pragma unroll
                                    for (int t = 0; t < 8; ++t) cw[t] = ld_shared_u32(g + 4u * t);
                                }
                                sw = ld_shared_u32(rowa + static_cast<uint32_t>(p.k >> 1) +
                                                   4u * static_cast<uint32_t>(u));
                            }
                            float sc[4];
                            e4m3x4_to_f32(sw, sc);
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const int v = region_dot(cw[2 * r], cw[2 * r + 1], &qv[jj][4 * r], corr[jj][r]);
                                acc[rr] = __fmaf_rn(__fmul_rn(sc[r], dd[jj][r >> 1]), static_cast<float>(v), acc[rr]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < RW; ++rr) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[rr] += __shfl_xor_sync(0xFFFFFFFFu, acc[rr], o);
            }
            if (lane < RW && row0 + lane < rows) {
                float v = acc[0];
#pragma unroll
                for (int rr = 1; rr < RW; ++rr)
                    if (lane == rr) v = acc[rr];
                p.dst[static_cast<int64_t>(mat) * p.rows_per_mat + r0 + row0 + lane] = bad ? nan : scale * v;
            }
            if (bad && warp == 0 && lane == 0) atomicOr(p.status, kDevBadPtr);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->empty[slot]);
        if ((r0 += SR) >= p.rows_per_mat) {
            r0 = 0;
            ++mat;
        }
        if (++slot == p.ring) {
            slot = 0;
            ph ^= 1u;
        }
    }
}

// Q8_1 blocks of 32 values, one warp per block: d = amax/127 and
// q = round-half-away(x * (1/d)), each step one float32 operation (q = 0
// when d = 0).
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float *__restrict__ x, int8_t *__restrict__ q,
                                                            float *__restrict__ d, int64_t nblocks) {
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; b < nblocks; b += wstride) {
        const float v = x[b * 32 + lane];
        float a = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
        const float db = q8_block_scale(a);
        const float id = q8_block_inv(db);
        q[b * 32 + lane] = static_cast<int8_t>(q8_code(v, id));
        if (lane == 0) d[b] = db;
    }
}

cudaError_t launch_quantize_q8_1(const float *x, int8_t *q, float *d, int64_t rows, int64_t k, int num_sms,
                                 cudaStream_t st) {
    const int64_t nblocks = rows * (k / 32);
    const int64_t want = (nblocks + 7) / 8;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8LL * num_sms)));
    return launch_pdl(quantize_q8_1_kernel, dim3(grid), dim3(256), 0, st, dim3(1, 1, 1), x, q, d, nblocks);
}

template <int F, int J, int RW, bool FX>
static cudaError_t launch_q8_j(const mq::Params &p, int num_sms, cudaStream_t st) {
    using namespace mq;
    const size_t smem = 128 + static_cast<size_t>(p.ring) * p.stage_bytes + sizeof(Ctl) + 16 +
                        (FX ? static_cast<size_t>(p.k / 64) * 72 : 0);
    cudaError_t e = cudaFuncSetAttribute(moe_q8_kernel<F, J, RW, FX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int grid = std::min(p.total_stages, num_sms);
    return launch_pdl(moe_q8_kernel<F, J, RW, FX>, dim3(grid), dim3(THREADS), smem, st, dim3(1, 1, 1), p);
}

template <int F, int RW, bool FX> static cudaError_t launch_q8_fx(const mq::Params &p, int num_sms, cudaStream_t st) {
    switch ((p.k / 64 + 31) / 32) {
    case 1: return launch_q8_j<F, 1, RW, FX>(p, num_sms, st);
    case 2: return launch_q8_j<F, 2, RW, FX>(p, num_sms, st);
    case 3: return launch_q8_j<F, 3, RW, FX>(p, num_sms, st);
    case 4: return launch_q8_j<F, 4, RW, FX>(p, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int F, int RW> static cudaError_t launch_q8_f(const mq::Params &p, int num_sms, cudaStream_t st) {
    return p.x ? launch_q8_fx<F, RW, true>(p, num_sms, st) : launch_q8_fx<F, RW, false>(p, num_sms, st);
}

cudaError_t launch_moe_q8(int dtype, const void *const *w_ptrs, int64_t rb, const float *scales, const int8_t *q,
                          const float *d, const float *x, float *dst, int64_t k, int64_t rows_per_mat, int mats,
                          int n_pairs, int n_used, int num_sms, uint32_t *status, uint64_t limit_ns, cudaStream_t st) {
    using namespace mq;
    if (k % 64 != 0 || k > QMM_Q8_MAX_K || rb % 4 != 0) return cudaErrorInvalidValue;
    Params p = {};
    p.w_ptrs = w_ptrs;
    p.scales = scales;
    p.q = q;
    p.d = d;
    p.x = x;
    p.dst = dst;
    p.k = k;
    p.rb = rb;
    p.rows_per_mat = static_cast<int>(rows_per_mat);
    p.mats = mats;
    p.n_pairs = n_pairs;
    p.n_used = n_used;
    // two rows per warp and stage when three such stages fit in shared memory
    // (more independent work per warp, half the per-row overhead), else one
    const int64_t budget = SMEM_BUDGET - static_cast<int64_t>(sizeof(Ctl)) - 256 - (x ? k / 64 * 72 : 0);
    const int rw = (budget / ((2 * COMPUTE_WARPS * rb + 15) / 16 * 16) >= 3) ? 2 : 1;
    const int sr = COMPUTE_WARPS * rw;
    p.stages_per_mat = static_cast<int>((rows_per_mat + sr - 1) / sr);
    p.total_stages = p.stages_per_mat * mats;
    p.stage_bytes = static_cast<int>((sr * rb + 15) / 16 * 16);
    p.ring = static_cast<int>(std::min<int64_t>(MAX_RING, budget / p.stage_bytes));
    if (p.ring < 2) return cudaErrorInvalidValue;
    p.status = status;
    p.limit_ns = limit_ns;
    switch (dtype * 2 + rw - 1) {
    case QMM_NVFP4 * 2: return launch_q8_f<QMM_NVFP4, 1>(p, num_sms, st);
    case QMM_NVFP4 * 2 + 1: return launch_q8_f<QMM_NVFP4, 2>(p, num_sms, st);
    case QMM_NVFP4_V2 * 2: return launch_q8_f<QMM_NVFP4_V2, 1>(p, num_sms, st);
    case QMM_NVFP4_V2 * 2 + 1: return launch_q8_f<QMM_NVFP4_V2, 2>(p, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
