// gemm_tc.cu -- the prefill GEMM dst[n][m] = sum_k W[m][k] X[n][k] on the
// 5th-generation tensor cores (tcgen05), for n > QMM_GEMV_MAX_N.
//
// The product is the one cera 0.4.0 examples/wgpu_gemm_bench.rs benchmarks
// (struct Shape; its mul_mat_reg_tile kernel decodes src0 blocks into shared
// memory with per-format loaders).  Here one CTA owns a 128 (m) x BN (n)
// output tile -- or two 128-row subtiles sharing every X stage (SUB = 2) --
// and a slice of k:
//
//   warp 0      raw-weight producer: the packed bytes of 256 k of all the
//               CTA's rows at a time into a ring of raw stages -- one 2-D TMA
//               box per stage over the rows viewed as 16-byte aligned row
//               groups (G rows when G*row_bytes is a multiple of 16), else
//               per-row 1-D bulk copies of 16-byte aligned supersets of each
//               row; with f32 weights (tf32 MMA, no decode) the W tiles, so
//               that two threads issue a stage's two 32 KB TMA requests;
//   warp 1      TMEM allocation and the single MMA-issuing thread:
//               tcgen05.mma.kind::f16, M=128, N=BN, K=16, sixteen per 256-wide
//               k stage, A (decoded W) read from tensor memory, B (X) from
//               shared memory, fp32 accumulators in BN TMEM columns per
//               subtile; tcgen05.commit releases the stages it read;
//   warp 2      X producer: the f16 copy of X through TMA with the 128-byte
//               swizzle -- one request per stage through a 3-D tensor map
//               ([k atoms][rows][atom]) when k allows, else one 2-D box per
//               128-byte k atom.  X is rounded once to f16 (round to nearest
//               even) by x_to_f16_kernel, like the cvt.rn.f16.f32 converter of
//               aprender-serve cublas_prefill/mod.rs;
//   warps 3-10  decode: thread = one W row = one TMEM lane (a warp owns the
//               lane quarter warp%4); the two warps of a quarter take the two
//               128-wide halves of every 256-wide k stage (SUB = 2: the two
//               subtiles), turn the row's raw bytes (raw stage in shared
//               memory) into f16 and write them into a ring of A slots in
//               tensor memory with tcgen05.st.  The decoded weights never
//               touch shared memory or HBM, so the shared-memory bandwidth is
//               left to the X stream and the raw bytes; then the same warps
//               run the epilogue: tcgen05.ld, the tile into shared memory as
//               [n][m], 32 columns at a time, each group leaving with a TMA
//               store while the next is read out of tensor memory.
//
// Stages are long on purpose: the issuing thread waits on mbarriers between
// stages, and a wait that follows tcgen05.commit costs a few hundred cycles,
// which sixteen queued MMAs (about a thousand cycles of tensor work) hide.
//
// f32 weights skip the decode: warp 2 loads W and X tiles as f32 with TMA and
// the MMA runs kind::tf32 (K=8, eight per 64-wide stage).
//
// Split-K: when the output has fewer tiles than the GPU has SMs, S CTAs of a
// thread-block cluster (dims 1 x 1 x S) share one output tile, each taking a
// contiguous share of the 256-wide k units.  Each writes its fp32 partial tile to its own shared
// memory; after a cluster barrier CTA z sums column slice z of all S partials
// through distributed shared memory in the fixed order 0..S-1 and stores it.
// No atomics: the result is deterministic.
//
// Every mbarrier wait is bounded by a wall-clock limit; a wait that runs out
// latches a status bit, the CTA stops issuing work, waits for its own copies
// and MMAs in flight, frees its tensor memory and returns (after the cluster
// barriers its peers also pass).
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

#include "decode.cuh"
#include "kernels.h"

namespace qmm {

namespace gemm {
constexpr int BM = 128;
constexpr int ATOM_ROW = 128;        // bytes of one operand row in one 128-byte swizzle atom
constexpr int RK = 256;              // k per raw-weight stage and per split-K unit
constexpr int NUM_DECODE_WARPS = 8;
constexpr int TMEM_MAX = 512;        // TMEM columns per SM
constexpr int WARP_RAW = 0, WARP_MMA = 1, WARP_X = 2, WARP_DEC0 = 3;
constexpr int THREADS = 32 * (WARP_DEC0 + NUM_DECODE_WARPS);  // 352
constexpr int MAX_SPLIT = 8;
constexpr int SMEM_LIMIT = 232448;   // 227 KB opt-in per CTA
constexpr int MAXS = 8;              // ring depth bound (barrier arrays)

struct Ctl {
    uint64_t b_full[MAXS], b_empty[MAXS];      // X (and f32 W) tiles
    uint64_t a_full[MAXS], a_empty[MAXS];      // decoded W tiles
    uint64_t raw_full[MAXS], raw_empty[MAXS];  // raw weight stages
    uint64_t accum;
    uint32_t tmem_base;
    int abort;
};

// Geometry of a (format, BN, SUB) instance: ring depths that fit in shared
// memory.  A CTA owns SUB 128-row subtiles (SUB = 2: two accumulators share
// every X stage, halving the X bytes per MMA).
template <int F, int BN, int SUB> struct Plan {
    static constexpr bool TF32 = (F == QMM_F32);
    static_assert(SUB == 1 || (SUB == 2 && !TF32), "two subtiles for packed W only");
    static constexpr int ROWS = BM * SUB;                  // W rows per CTA
    static constexpr int QK = Fmt<F>::QK, BB = Fmt<F>::BB;
    // k per MMA stage: packed W takes 256/SUB (16 MMAs of K=16 per stage
    // across the subtiles); f32 W takes 64 (8 MMAs of K=8)
    static constexpr int KPS = TF32 ? 64 : RK / SUB;
    static constexpr int ELEM = TF32 ? 4 : 2;
    static constexpr int ATOMS = KPS * ELEM / ATOM_ROW;   // swizzle atoms along k per stage
    static constexpr int KMMA = TF32 ? 8 : 16;
    static constexpr int MMAS = KPS / KMMA;               // MMAs per stage and subtile
    static constexpr int B_ATOM = BN * ATOM_ROW;
    static constexpr int B_STAGE = ATOMS * B_ATOM;
    static constexpr int A_ATOM = BM * ATOM_ROW;
    static constexpr int A_STAGE = TF32 ? ATOMS * A_ATOM : 0;  // f32 W tiles in shared memory
    // raw stage: 256 k of every row; pitch an odd multiple of 16 bytes >= the
    // row bytes plus the largest misalignment (block rows are 2-byte aligned)
    static constexpr int RB = TF32 ? 0 : RK / QK * BB;
    static constexpr int SLACK = (F == QMM_Q4_K) ? 0 : ((F == QMM_NVFP4) ? 12 : 14);
    static constexpr int P0 = TF32 ? 16 : (RB + SLACK + 15) / 16 * 16;
    static constexpr int P = ((P0 / 16) % 2 == 1) ? P0 : P0 + 16;
    static constexpr int RAW_STAGE = TF32 ? 0 : ROWS * P;
    static constexpr int CTL = static_cast<int>(sizeof(Ctl));
    // raw stages: three when that still leaves 128 KB for X stages, else two
    static constexpr int RS = TF32 ? 0 : ((SMEM_LIMIT - 1024 - CTL - 3 * RAW_STAGE >= 131072) ? 3 : 2);
    static constexpr int AVAIL = SMEM_LIMIT - 1024 - CTL - RS * RAW_STAGE;
    // X (and f32 W) stages: as many as fit, at most MAXS
    static constexpr int BS0 = AVAIL / (B_STAGE + A_STAGE);
    static constexpr int BS = BS0 > MAXS ? MAXS : BS0;
    // decoded-W (A) stages: packed W in tensor memory after the SUB
    // accumulators (SUB * KPS/2 columns each: two f16 per column, subtile t at
    // +64t); f32 W with the X stages
    static constexpr int D_COLS = SUB * BN;
    static constexpr int A_COLS = SUB * KPS / 2;
    static constexpr int AS0 = TF32 ? BS : (TMEM_MAX - D_COLS) / A_COLS;
    static constexpr int AS = AS0 > MAXS ? MAXS : AS0;
    static constexpr int RING = BS * (B_STAGE + A_STAGE) + RS * RAW_STAGE;
    static constexpr int TMEM_COLS = TF32 ? BN : TMEM_MAX;
    static constexpr int RED = ROWS * BN * 4;             // split-K partial tile (aliases the rings)
    static constexpr int BODY = RING > RED ? RING : RED;
    static constexpr size_t SMEM = 1024 + BODY + sizeof(Ctl);
    static_assert(TF32 || RS >= 2, "raw ring needs two stages");
    static_assert(BS >= 2 && AS >= 2, "rings need two stages");
    static_assert(TF32 || D_COLS + AS * A_COLS <= TMEM_MAX, "A slots exceed tensor memory");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS >= 32 && TMEM_COLS <= 512, "TMEM allocation");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory plan too large");
    static constexpr uint32_t IDESC = mma_idesc(TF32 ? 2u : 0u, BM, BN);
};
}  // namespace gemm

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

struct GemmParams {
    const uint8_t *w;
    int64_t rb;
    float *dst;
    int M, N, K;
    int units;   // 256-wide k units: ceil(K / 256)
    int w_early; // 1: the kernel before this one only wrote the f16 copy of X, so W may be read before it ends
    int raw_g;   // rows per 16-byte-aligned row group of the raw-weight tensor map; 0 = per-row bulk copies
    int splits;  // CTAs per output tile (cluster size along z)
    int x3d;     // 1: X (and f32 W) maps are 3-D [k atoms][rows][atom]: one TMA request per stage
    int dtma;    // 1: the tile is stored with TMA stores through tmap_d (m % 4 == 0)
    uint32_t *status;
    uint64_t limit_ns;
    int debug_skip;
};

template <int F, int BN, int SUB>
__global__ void __launch_bounds__(gemm::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_raw, const __grid_constant__ CUtensorMap tmap_d,
                   const GemmParams p) {
    using namespace gemm;
    using PL = Plan<F, BN, SUB>;
    constexpr bool TF32 = PL::TF32;
    constexpr int KPS = PL::KPS, BS = PL::BS, AS = PL::AS, RS = PL::RS, ROWS = PL::ROWS;
    constexpr int SPU = RK / KPS;  // MMA stages per 256-wide unit

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sB = base;
    uint8_t *sA = sB + BS * PL::B_STAGE;  // f32 W only
    uint8_t *sRaw = sA + BS * PL::A_STAGE;
    float *sRed = reinterpret_cast<float *>(base);  // split-K partial, after the main loop
    Ctl *ctl = reinterpret_cast<Ctl *>(base + PL::BODY);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * ROWS, n0 = blockIdx.y * BN;
    const int S = p.splits;
    const int z = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int u0 = z * p.units / S, u1 = (z + 1) * p.units / S;
    const int KT = (p.K + KPS - 1) / KPS;
    const int kt0 = u0 * SPU;
    const int kt1 = min(u1 * SPU, KT);
    const int NK = kt1 - kt0;  // MMA stages of this CTA (>= 1)

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAXS; ++s) {
            mbar_init(&ctl->b_full[s], TF32 ? 2 : 1);  // f32 W: the W and X producers each arrive
            mbar_init(&ctl->b_empty[s], 1);
            mbar_init(&ctl->a_full[s], NUM_DECODE_WARPS);
            mbar_init(&ctl->a_empty[s], 1);
            mbar_init(&ctl->raw_full[s], 1);
            mbar_init(&ctl->raw_empty[s], NUM_DECODE_WARPS);
        }
        mbar_init(&ctl->accum, 1);
        ctl->abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmap_x);
        if (TF32) prefetch_tensormap(&tmap_w);
        if (!TF32 && p.raw_g > 0) prefetch_tensormap(&tmap_raw);
        // weights that may be read before the kernel in front ends: the first
        // ring of raw stages goes out now, before the TMEM allocation and the
        // block-wide barrier (this thread is the raw producer's issuing lane)
        if constexpr (!TF32) {
            const int npre = (p.w_early && p.raw_g > 0) ? min(RS, u1 - u0) : 0;
            for (int i = 0; i < npre; ++i) {
                const int64_t seg_off = static_cast<int64_t>(u0 + i) * PL::RB;
                const int G = p.raw_g;
                mbar_arrive_expect_tx(&ctl->raw_full[i], ROWS * PL::P);
                for (int g = 0; g < G; ++g) {
                    const int64_t xb = (static_cast<int64_t>(g) * p.rb + seg_off) & ~int64_t(15);
                    tma_load_2d(sRaw + i * PL::RAW_STAGE + g * (ROWS / G) * PL::P, &tmap_raw,
                                static_cast<int32_t>(xb / 2), m0 / G, &ctl->raw_full[i]);
                }
            }
        }
    }
    if (warp == WARP_MMA) {
        tmem_alloc(&ctl->tmem_base, PL::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort;
    // Everything below may touch memory the previous kernel in the stream
    // wrote.  When that kernel is x_to_f16_kernel (w_early), it wrote only the
    // f16 copy of X, which the X producer alone reads: the other roles go
    // ahead (weights, decode, MMA on stages the X producer has released), and
    // the epilogue's stores follow the X loads through the barriers anyway.
    if (!p.w_early || warp == WARP_X) griddep_wait();

    if (warp == WARP_RAW) {
        // ------------- raw weight producer (all 32 lanes); f32 W: the W tiles -------------
        if constexpr (TF32) {
            if (lane == 0) {
                int last[BS];
#pragma unroll
                for (int s = 0; s < BS; ++s) last[s] = -1;
                for (int i = 0; i < NK; ++i) {
                    const int kt = kt0 + i, s = i % BS;
                    const uint32_t ph = (i / BS) & 1;
                    if (!mbar_wait_bounded(&ctl->b_empty[s], ph ^ 1, abort, p.status, p.limit_ns)) break;
                    mbar_arrive_expect_tx(&ctl->b_full[s], PL::A_STAGE);
                    if (p.x3d) {
                        tma_load_3d(sA + s * PL::A_STAGE, &tmap_w, 0, m0, kt * PL::ATOMS, &ctl->b_full[s]);
                    } else {
#pragma unroll
                        for (int j = 0; j < PL::ATOMS; ++j) {
                            const int kx = kt * KPS + j * (ATOM_ROW / PL::ELEM);
                            tma_load_2d(sA + s * PL::A_STAGE + j * PL::A_ATOM, &tmap_w, kx, m0, &ctl->b_full[s]);
                        }
                    }
                    last[s] = i;
                }
                if (*abort) {
                    for (int s = 0; s < BS; ++s)
                        if (last[s] >= 0) mbar_wait_drain(&ctl->b_full[s], (last[s] / BS) & 1, p.status, p.limit_ns);
                }
            }
            __syncwarp();
        }
        if constexpr (!TF32) {
            int last[RS];
#pragma unroll
            for (int r = 0; r < RS; ++r) last[r] = -1;
            const int npre = (p.w_early && p.raw_g > 0) ? min(RS, u1 - u0) : 0;  // issued in the prologue
            for (int i = 0; u0 + i < u1; ++i) {
                const int u = u0 + i, r = i % RS;
                const uint32_t ph = (i / RS) & 1;
                if (i < npre) {
                    last[r] = i;
                    continue;
                }
                const bool ok = mbar_wait_bounded(&ctl->raw_empty[r], ph ^ 1, abort, p.status, p.limit_ns);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                const int64_t seg_off = static_cast<int64_t>(u) * PL::RB;
                uint8_t *stage = sRaw + r * PL::RAW_STAGE;
                if (p.raw_g > 0) {
                    // one 2-D TMA box per row residue g: rows m0+g, m0+g+G, ... land
                    // contiguously at slots g*(ROWS/G) ... with pitch P
                    if (lane == 0) {
                        const int G = p.raw_g;
                        mbar_arrive_expect_tx(&ctl->raw_full[r], ROWS * PL::P);
                        for (int g = 0; g < G; ++g) {
                            const int64_t xb = (static_cast<int64_t>(g) * p.rb + seg_off) & ~int64_t(15);
                            tma_load_2d(stage + g * (ROWS / G) * PL::P, &tmap_raw, static_cast<int32_t>(xb / 2),
                                        m0 / G, &ctl->raw_full[r]);
                        }
                    }
                    __syncwarp();
                    last[r] = i;
                    continue;
                }
                const int len = static_cast<int>(min(static_cast<int64_t>(PL::RB), p.rb - seg_off));
                uint32_t bytes[ROWS / 32];
                const uint8_t *src[ROWS / 32];
                uint32_t tot = 0;
#pragma unroll
                for (int j = 0; j < ROWS / 32; ++j) {
                    const int row = lane + 32 * j, gm = m0 + row;
                    bytes[j] = 0;
                    src[j] = nullptr;
                    if (gm < p.M) {
                        const uint8_t *s0 = p.w + static_cast<int64_t>(gm) * p.rb + seg_off;
                        const uintptr_t a = reinterpret_cast<uintptr_t>(s0) & ~uintptr_t(15);
                        const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(s0) - a);
                        src[j] = reinterpret_cast<const uint8_t *>(a);
                        bytes[j] = (mis + len + 15u) & ~15u;
                        tot += bytes[j];
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
                if (lane == 0) mbar_arrive_expect_tx(&ctl->raw_full[r], tot);
                __syncwarp();
#pragma unroll
                for (int j = 0; j < ROWS / 32; ++j)
                    if (bytes[j]) bulk_load_1d(stage + (lane + 32 * j) * PL::P, src[j], bytes[j], &ctl->raw_full[r]);
                last[r] = i;
            }
            if (lane == 0 && *abort) {
                for (int r = 0; r < RS; ++r)
                    if (last[r] >= 0) mbar_wait_drain(&ctl->raw_full[r], (last[r] / RS) & 1, p.status, p.limit_ns);
            }
            __syncwarp();
        }
    } else if (warp == WARP_X) {
        // ------------- X (and f32 W) tile producer -------------
        if (lane == 0) {
            int last[BS];
#pragma unroll
            for (int s = 0; s < BS; ++s) last[s] = -1;
            for (int i = 0; i < NK; ++i) {
                const int kt = kt0 + i, s = i % BS;
                const uint32_t ph = (i / BS) & 1;
                if (!mbar_wait_bounded(&ctl->b_empty[s], ph ^ 1, abort, p.status, p.limit_ns)) break;
                if (p.debug_skip && i == 0) continue;  // test hook: stage 0 never fills
                mbar_arrive_expect_tx(&ctl->b_full[s], PL::B_STAGE);
                if (p.x3d) {
                    // the whole stage (every 128-byte k atom of the tile rows) in one request:
                    // one SM's TMA engine spends about the same time per request up to 32 KB
                    tma_load_3d(sB + s * PL::B_STAGE, &tmap_x, 0, n0, kt * PL::ATOMS, &ctl->b_full[s]);
                } else {
#pragma unroll
                    for (int j = 0; j < PL::ATOMS; ++j) {
                        const int kx = kt * KPS + j * (ATOM_ROW / PL::ELEM);
                        tma_load_2d(sB + s * PL::B_STAGE + j * PL::B_ATOM, &tmap_x, kx, n0, &ctl->b_full[s]);
                    }
                }
                last[s] = i;
            }
            if (*abort) {
                for (int s = 0; s < BS; ++s)
                    if (last[s] >= 0) mbar_wait_drain(&ctl->b_full[s], (last[s] / BS) & 1, p.status, p.limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------- MMA issuer -------------
        if (lane == 0) {
            for (int i = 0; i < NK; ++i) {
                const int sb = i % BS, sa = i % AS;
                if (!mbar_wait_bounded(&ctl->b_full[sb], (i / BS) & 1, abort, p.status, p.limit_ns)) break;
                if (!TF32 && !mbar_wait_bounded(&ctl->a_full[sa], (i / AS) & 1, abort, p.status, p.limit_ns)) break;
                tc_fence_after();
                const uint32_t b_addr = smem_u32(sB + sb * PL::B_STAGE);
#pragma unroll
                for (int t = 0; t < SUB; ++t) {  // subtiles share every X stage
#pragma unroll
                    for (int kk = 0; kk < PL::MMAS; ++kk) {
                        // K step kk: atom kk/4, 32 bytes (16 f16 or 8 f32) per step inside the atom
                        const uint32_t off = static_cast<uint32_t>((kk >> 2) * PL::B_ATOM + 32 * (kk & 3));
                        const uint64_t bd = sw128_desc(b_addr + off);
                        if constexpr (TF32) {
                            const uint32_t aoff = static_cast<uint32_t>((kk >> 2) * PL::A_ATOM + 32 * (kk & 3));
                            const uint64_t ad = sw128_desc(smem_u32(sA + sa * PL::A_STAGE) + aoff);
                            mma_tf32(tmem, ad, bd, PL::IDESC, (i | kk) != 0);
                        } else {
                            // A slot sa after the accumulators: subtile t at +64t, 8 columns per K=16 step
                            const uint32_t at =
                                tmem + PL::D_COLS + static_cast<uint32_t>(sa * PL::A_COLS + 64 * t + 8 * kk);
                            mma_f16_tmem_a(tmem + static_cast<uint32_t>(t * BN), at, bd, PL::IDESC, (i | kk) != 0);
                        }
                    }
                }
                mma_commit(&ctl->b_empty[sb]);
                if (!TF32) mma_commit(&ctl->a_empty[sa]);
            }
            mma_commit(&ctl->accum);  // arrives once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // ------------- decode warps -------------
        // Thread = one W row = one TMEM lane (lane quarter warp%4).  SUB == 1:
        // warps 3-6 decode the first 128 k of every 256-wide stage, warps 7-10
        // the second.  SUB == 2: warps 3-6 decode subtile 0 (rows 0-127),
        // warps 7-10 subtile 1, each the whole 128-wide stage.
        if constexpr (!TF32) {
            constexpr int SPU_ = RK / KPS;  // MMA stages per raw unit (= SUB)
            const int q = warp & 3;
            const int hh = (warp - WARP_DEC0) >> 2;
            const int row = (SUB == 2 ? 128 * hh : 0) + 32 * q + lane;
            const int slot = (p.raw_g > 0) ? (row % p.raw_g) * (ROWS / p.raw_g) + row / p.raw_g : row;
            const uint32_t rowoff = static_cast<uint32_t>(slot * PL::P);
            const int gm = m0 + row;
            const uint32_t misb = static_cast<uint32_t>(
                (reinterpret_cast<uintptr_t>(p.w) + static_cast<int64_t>(gm < p.M ? gm : 0) * p.rb) & 15u);
            const uint32_t raw0 = smem_u32(sRaw);
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + PL::D_COLS + 64u * hh;
            for (int i = 0; i < NK; ++i) {
                const int kt = kt0 + i, sa = i % AS;
                const int unit = kt / SPU_, ui = unit - u0, r = ui % RS;
                if (kt % SPU_ == 0) {
                    const bool ok = mbar_wait_bounded(&ctl->raw_full[r], (ui / RS) & 1, abort, p.status, p.limit_ns);
                    if (!__all_sync(0xFFFFFFFFu, ok)) break;
                }
                const bool ok = mbar_wait_bounded(&ctl->a_empty[sa], ((i / AS) & 1) ^ 1, abort, p.status, p.limit_ns);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                const uint32_t mis = (misb + static_cast<uint32_t>(unit * PL::RB)) & 15u;
                const uint32_t src = raw0 + static_cast<uint32_t>(r * PL::RAW_STAGE) + rowoff + mis;
                const int H = (SUB == 2) ? (kt % SPU_) : hh;  // which 128-wide half of the unit
                uint32_t o[64];
                constexpr bool kAligned = (F == QMM_Q4_0 || F == QMM_Q8_0 || F == QMM_NVFP4);
                if (kAligned && mis == 0 && gm < p.M && static_cast<int64_t>(unit) * RK + 128 * H + 128 <= p.K) {
                    // 16-byte aligned segment: conflict-free 16-byte loads, static offsets
                    if (H == 0)
                        Dec128<F, 0>::run(src, o);
                    else
                        Dec128<F, 1>::run(src, o);
                } else {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int e0 = 128 * H + 32 * t;  // weights within the 256-wide unit
                        uint32_t ot[16];
                        if (gm < p.M && static_cast<int64_t>(unit) * RK + e0 < p.K) {
                            decode32_s<F>(src, e0, ot);
                        } else {
#pragma unroll
                            for (int q2 = 0; q2 < 16; ++q2) ot[q2] = 0u;
                        }
#pragma unroll
                        for (int q2 = 0; q2 < 16; ++q2) o[16 * t + q2] = ot[q2];
                    }
                }
                tmem_st_32x32b_x64(tq + static_cast<uint32_t>(sa * PL::A_COLS), o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctl->a_full[sa]);
                    // the last stage of a raw unit (or of this CTA) frees the raw stage
                    if (kt % SPU_ == SPU_ - 1 || i == NK - 1) mbar_arrive(&ctl->raw_empty[r]);
                }
            }
        }
    }

    // ---------------- epilogue ----------------
    const bool is_epi = warp >= WARP_DEC0;
    bool have = false;
    if (is_epi) {
        const bool drained = mbar_wait_drain(&ctl->accum, 0, p.status, p.limit_ns);
        // the next kernel in the stream may launch now: its launch and start-up
        // overlap this epilogue, and its CTAs do not sit waiting through the main loop
        if (warp == WARP_DEC0 && lane == 0) griddep_launch();
        if (!drained) *abort = 1;
        have = __all_sync(0xFFFFFFFFu, drained && !*abort);  // tcgen05.ld is warp-collective
    }
    // Warp (quarter q, half hh) stores: SUB == 1: rows 32q+lane, columns
    // [BN/2*hh, BN/2*hh + BN/2); SUB == 2: rows 128hh + 32q + lane (subtile hh,
    // accumulator at TMEM column BN*hh), all BN columns.
    const int q = warp & 3;                                           // TMEM lane quarter of this warp
    const int hh = (warp >= WARP_DEC0 + 4) ? 1 : 0;
    constexpr int ECOLS = (SUB == 2) ? BN : BN / 2;                   // output columns per warp
    const int colbase = (SUB == 2) ? 0 : (BN / 2) * hh;               // first output column in the tile
    const uint32_t dcol = static_cast<uint32_t>((SUB == 2) ? BN * hh : (BN / 2) * hh);  // its TMEM column
    const int rloc = (SUB == 2 ? 128 * hh : 0) + 32 * q + lane;      // tile row of this thread
    if (S == 1 && p.dtma) {
        // tile -> shared memory as [BN][ROWS] (m contiguous), 32 columns at a
        // time; each finished group of columns leaves with a TMA store while
        // the next is read out of tensor memory
        if (is_epi) {
            if (have) tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < ECOLS / 32; ++c) {
                if (have) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + dcol + 32 * c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) sRed[(colbase + 32 * c + j) * ROWS + rloc] = __uint_as_float(v[j]);
                }
                fence_proxy_async_smem();  // the generic-proxy writes above, before the async-proxy read
                asm volatile("bar.sync 1, %0;" ::"r"(32 * NUM_DECODE_WARPS) : "memory");  // every epilogue warp
                if (warp == WARP_DEC0 && lane == 0 && !*abort) {
                    // columns 32c.. of each column half (SUB == 1) or of the tile (SUB == 2)
                    for (int h2 = 0; h2 < (SUB == 2 ? 1 : 2); ++h2) {
                        const int col = (SUB == 2 ? 0 : (BN / 2) * h2) + 32 * c;
                        tma_store_2d(&tmap_d, m0, n0 + col, sRed + col * ROWS);
                    }
                    bulk_commit_group();
                }
            }
            if (warp == WARP_DEC0 && lane == 0 && !*abort) bulk_wait_group_read0();  // sources valid until read
        }
    } else if (S == 1) {
        if (is_epi && have) {
            tc_fence_after();
            const int gm = m0 + rloc;
#pragma unroll 1
            for (int c = 0; c < ECOLS / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + dcol + 32 * c, v);
                tmem_ld_wait();
                const int gn0 = n0 + colbase + 32 * c;
                if (gm < p.M) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (gn0 + j < p.N) p.dst[static_cast<int64_t>(gn0 + j) * p.M + gm] = __uint_as_float(v[j]);
                }
            }
        }
    } else {
        // partial tile -> own shared memory, column-major [BN][ROWS]
        if (is_epi && have) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < ECOLS / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + dcol + 32 * c, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) sRed[(colbase + 32 * c + j) * ROWS + rloc] = __uint_as_float(v[j]);
            }
        }
        __syncwarp();
        cluster_sync_all();
        // a CTA that gave up left no valid partial: then nobody stores
        int any_abort = 0;
        for (int pr = 0; pr < S; ++pr) any_abort |= ld_dsmem_u32(mapa_shared(smem_u32(&ctl->abort), pr));
        // CTA z sums column slice z of the S partials in rank order and stores it
        splitk_reduce_store<ROWS>(smem_u32(sRed), S, z, BN, m0, n0, p.M, p.N, p.dst,
                                             static_cast<int>(threadIdx.x), THREADS, any_abort != 0);
        __syncwarp();
        cluster_arrive_relaxed_wait();  // peers keep their partials until every slice is read
    }
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// X [n][k] f32 -> [n][k] f16, round to nearest even; k % 8 == 0.  At most
// two CTAs per SM, so that the GEMM CTAs launched behind it fit next to them
// and stage and decode their first weights while it runs; four 32-byte
// chunks in flight per thread.
constexpr int X16_THREADS = 256, X16_CTAS_PER_SM = 2;
__device__ __forceinline__ void x16_chunk(const float *__restrict__ x, __half *__restrict__ x16, int64_t i) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(x) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4 *>(x) + 2 * i + 1);
    const __half2 h0 = __floats2half2_rn(a.x, a.y), h1 = __floats2half2_rn(a.z, a.w);
    const __half2 h2 = __floats2half2_rn(b.x, b.y), h3 = __floats2half2_rn(b.z, b.w);
    reinterpret_cast<uint4 *>(x16)[i] = make_uint4(h2_bits(h0), h2_bits(h1), h2_bits(h2), h2_bits(h3));
}
__global__ void __launch_bounds__(X16_THREADS) x_to_f16_kernel(const float *__restrict__ x, __half *__restrict__ x16,
                                                               int64_t total8) {
    griddep_wait();    // X may come from the kernel before this one; X16 may still be read by it
    griddep_launch();  // the GEMM may start staging weights while this runs
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < total8; i += 4 * stride) {
        float4 a[4], b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            a[u] = __ldg(reinterpret_cast<const float4 *>(x) + 2 * (i + u * stride));
            b[u] = __ldg(reinterpret_cast<const float4 *>(x) + 2 * (i + u * stride) + 1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const __half2 h0 = __floats2half2_rn(a[u].x, a[u].y), h1 = __floats2half2_rn(a[u].z, a[u].w);
            const __half2 h2 = __floats2half2_rn(b[u].x, b[u].y), h3 = __floats2half2_rn(b[u].z, b[u].w);
            reinterpret_cast<uint4 *>(x16)[i + u * stride] =
                make_uint4(h2_bits(h0), h2_bits(h1), h2_bits(h2), h2_bits(h3));
        }
    }
    for (; i < total8; i += stride) x16_chunk(x, x16, i);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// 2-D tiled map over a row-major [rows][cols] matrix, box [box_rows][box_cols],
// 128-byte swizzle (box_cols * elem == 128), zero fill outside the matrix.
static bool make_map(CUtensorMap *map, const void *ptr, CUtensorMapDataType dt, int elem, int64_t rows, int64_t cols,
                     int box_rows, int box_cols) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a row-major [rows][cols] matrix as [cols/A][rows][A] with A the
// elements of one 128-byte swizzle atom (the atom index outermost, stride 128
// bytes): a box [A][box_rows][atoms] lands as `atoms` consecutive
// [box_rows x 128 B] swizzled atoms, i.e. one request per pipeline stage.
// Needs cols % A == 0 (else the last atom of a row would alias the next row).
static bool make_map_3d(CUtensorMap *map, const void *ptr, CUtensorMapDataType dt, int elem, int64_t rows,
                        int64_t cols, int box_rows, int atoms) {
    auto fn = get_encode_fn();
    const int A = 128 / elem;
    if (!fn || cols % A != 0) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(A), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(cols / A)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * elem, 128};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(A), static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(atoms)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raw packed-weight map: the [m][rb] bytes viewed as [m/G][G*rb/2] uint16 with
// G the smallest row group whose byte stride is a multiple of 16; boxes of
// [rows/G][P/2] (P bytes per row, no swizzle; `rows` W rows per CTA).  Returns
// G, or 0 when no such view exists (then the kernel copies row by row).
static int make_raw_map(CUtensorMap *map, const void *w, int64_t m, int64_t rb, int pitch, int rows) {
    auto fn = get_encode_fn();
    if (!fn) return 0;
    int G = 1;
    while (G <= 8 && (G * rb) % 16 != 0) G *= 2;
    if (G > 8 || m % G != 0 || pitch % 16 != 0 || pitch / 2 > 256) return 0;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(G * rb / 2), static_cast<cuuint64_t>(m / G)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(G * rb)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(pitch / 2), static_cast<cuuint32_t>(rows / G)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(w), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? G : 0;
}

template <int F, int BN, int SUB> static cudaError_t set_attr() {
    return cudaFuncSetAttribute(gemm_tc_kernel<F, BN, SUB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(gemm::Plan<F, BN, SUB>::SMEM));
}

// Opt every instance into its shared-memory carve-out; called once per device
// (with that device current) when a handle is created.
cudaError_t gemm_tc_init() {
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
    };
    chk(set_attr<QMM_F32, 128, 1>());
    chk(set_attr<QMM_Q4_0, 128, 1>());
    chk(set_attr<QMM_Q8_0, 128, 1>());
    chk(set_attr<QMM_Q4_K, 128, 1>());
    chk(set_attr<QMM_Q6_K, 128, 1>());
    chk(set_attr<QMM_NVFP4, 128, 1>());
    chk(set_attr<QMM_Q4_0, 128, 2>());
    chk(set_attr<QMM_Q8_0, 128, 2>());
    chk(set_attr<QMM_Q4_K, 128, 2>());
    chk(set_attr<QMM_Q6_K, 128, 2>());
    chk(set_attr<QMM_NVFP4, 128, 2>());
    return e;
}

// Split count: enough CTAs per output tile to cover the SMs, at most one per
// 256-wide k unit, a power of two up to 8 (it must divide the tile width).
static int choose_splits(int64_t tiles, int units, int num_sms) {
    int s = 1;
    while (s < gemm::MAX_SPLIT && tiles * (s * 2) <= num_sms && s * 2 <= units) s *= 2;
    return s;
}

template <int F, int SUB>
static cudaError_t launch_sub(const GemmArgs &a, GemmParams p, int num_sms, cudaStream_t st) {
    using namespace gemm;
    constexpr int BN = 128;
    using PL = Plan<F, BN, SUB>;
    CUtensorMap map_x, map_w, map_raw;
    memset(&map_w, 0, sizeof(map_w));
    memset(&map_raw, 0, sizeof(map_raw));
    const void *xsrc = (F == QMM_F32) ? static_cast<const void *>(a.x) : a.x16;
    const CUtensorMapDataType xdt = (F == QMM_F32) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    p.x3d = make_map_3d(&map_x, xsrc, xdt, PL::ELEM, a.n, a.k, BN, PL::ATOMS) &&
            (F != QMM_F32 || make_map_3d(&map_w, a.w, xdt, PL::ELEM, a.m, a.k, BM, PL::ATOMS));
    if (!p.x3d) {
        if (!make_map(&map_x, xsrc, xdt, PL::ELEM, a.n, a.k, BN, ATOM_ROW / PL::ELEM)) return cudaErrorInvalidValue;
        if (F == QMM_F32 && !make_map(&map_w, a.w, xdt, PL::ELEM, a.m, a.k, BM, ATOM_ROW / PL::ELEM))
            return cudaErrorInvalidValue;
    }
    if (F != QMM_F32) map_w = map_x;  // unused by the packed-format kernels
    p.raw_g = (F == QMM_F32) ? 0 : make_raw_map(&map_raw, a.w, a.m, a.rb, PL::P, PL::ROWS);
    const int64_t m_tiles = (a.m + PL::ROWS - 1) / PL::ROWS, n_tiles = (a.n + BN - 1) / BN;
    p.splits = choose_splits(m_tiles * n_tiles, p.units, num_sms);
    // dst [n][m] f32 viewed by a TMA store map: boxes of [BN n][ROWS m]
    CUtensorMap map_d;
    memset(&map_d, 0, sizeof(map_d));
    p.dtma = 0;
    if (a.m % 4 == 0) {
        auto fn = get_encode_fn();
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.m), static_cast<cuuint64_t>(a.n)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.m) * 4};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(PL::ROWS), 32u};
        const cuuint32_t estr[2] = {1, 1};
        p.dtma = fn && fn(&map_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.dst, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const dim3 grid(static_cast<unsigned>(m_tiles), static_cast<unsigned>(n_tiles), static_cast<unsigned>(p.splits));
    const dim3 cluster(1, 1, static_cast<unsigned>(p.splits));
    return launch_pdl(gemm_tc_kernel<F, BN, SUB>, grid, dim3(THREADS), PL::SMEM, st, cluster, map_x, map_w, map_raw,
                      map_d, p);
}

template <int F>
static cudaError_t launch_gemm_t(const GemmArgs &a, int num_sms, cudaStream_t st) {
    using namespace gemm;
    constexpr int BN = 128;
    bool pdl = false;
    if (F != QMM_F32) {
        const int64_t total8 = a.n * a.k / 8;
        const int64_t want = (total8 + X16_THREADS - 1) / X16_THREADS;
        const int64_t cap = static_cast<int64_t>(X16_CTAS_PER_SM) * num_sms;
        const int grid = static_cast<int>(want < cap ? want : cap);
        cudaError_t e = launch_pdl(x_to_f16_kernel, dim3(grid), dim3(X16_THREADS), 0, st, dim3(1, 1, 1), a.x,
                                   static_cast<__half *>(a.x16), total8);
        if (e != cudaSuccess) return e;
        pdl = true;
    }
    GemmParams p;
    p.w = static_cast<const uint8_t *>(a.w);
    p.rb = a.rb;
    p.dst = a.dst;
    p.M = static_cast<int>(a.m);
    p.N = static_cast<int>(a.n);
    p.K = static_cast<int>(a.k);
    p.units = static_cast<int>((a.k + RK - 1) / RK);
    p.raw_g = 0;
    p.w_early = pdl ? 1 : 0;
    p.splits = 1;
    p.x3d = 0;
    p.status = a.status;
    p.limit_ns = a.wait_limit_ns;
    p.debug_skip = a.debug_skip_first_b_load;
    if constexpr (F != QMM_F32) {
        // two 128-row subtiles per CTA halve the X bytes per MMA; take them
        // when they cover the SMs as well without more split-K (whose partial
        // reduction costs more than the X traffic it saves)
        const int64_t n_tiles = (a.n + BN - 1) / BN;
        const int64_t t1 = (a.m + BM - 1) / BM * n_tiles, t2 = (a.m + 2 * BM - 1) / (2 * BM) * n_tiles;
        const int s1 = choose_splits(t1, p.units, num_sms), s2 = choose_splits(t2, p.units, num_sms);
        if (s2 <= s1 && t2 * s2 >= std::min<int64_t>(t1 * s1, num_sms)) return launch_sub<F, 2>(a, p, num_sms, st);
    }
    return launch_sub<F, 1>(a, p, num_sms, st);
}

cudaError_t launch_gemm_tc(const GemmArgs &a, int num_sms, cudaStream_t st) {
    switch (a.dtype) {
    case QMM_F32: return launch_gemm_t<QMM_F32>(a, num_sms, st);
    case QMM_Q4_0: return launch_gemm_t<QMM_Q4_0>(a, num_sms, st);
    case QMM_Q8_0: return launch_gemm_t<QMM_Q8_0>(a, num_sms, st);
    case QMM_Q4_K: return launch_gemm_t<QMM_Q4_K>(a, num_sms, st);
    case QMM_Q6_K: return launch_gemm_t<QMM_Q6_K>(a, num_sms, st);
    case QMM_NVFP4: return launch_gemm_t<QMM_NVFP4>(a, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
