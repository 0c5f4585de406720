// common.cuh -- shared device helpers of the qmm CUDA library (sm_103a only).
//
// Hand-written inline PTX for the Blackwell data movers and tensor cores:
// mbarrier waits with a time limit, 1-D/2-D bulk tensor copies (TMA), and the
// tcgen05 family (TMEM alloc/dealloc, MMA, commit, TMEM loads).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qmm.h"

namespace qmm {

// Device status bits written into the handle's status word.
constexpr uint32_t kDevTimeout = 1u;   // a bounded wait ran out
constexpr uint32_t kDevBadPtr = 2u;    // a device-side pointer (MoE table entry) was null or misaligned

// Format traits: QK weights per block, BB bytes per block.
template <int F> struct Fmt;
template <> struct Fmt<QMM_F32> { static constexpr int QK = 1, BB = 4; };
template <> struct Fmt<QMM_Q4_0> { static constexpr int QK = 32, BB = 18; };
template <> struct Fmt<QMM_Q8_0> { static constexpr int QK = 32, BB = 34; };
template <> struct Fmt<QMM_Q4_K> { static constexpr int QK = 256, BB = 144; };
template <> struct Fmt<QMM_Q6_K> { static constexpr int QK = 256, BB = 210; };
template <> struct Fmt<QMM_NVFP4> { static constexpr int QK = 64, BB = 36; };

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the barrier's phase with this parity has completed.  Gives up
// when *abort becomes nonzero (another role gave up) or after limit_ns of
// wall time; on the time limit it latches kDevTimeout in *status, raises
// *abort and returns false.  Never traps.  The common case -- the phase has
// already completed -- is one try_wait inline; the polling loop lives out of
// line (a long inlined loop next to tcgen05.mma issue slowed the issuing
// thread several-fold).
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                   uint32_t *status, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  uint32_t *status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort, status, limit_ns);
}

// Programmatic dependent launch: every kernel of the library is launched with
// the programmatic-serialization attribute, so it may start while the kernel
// before it in the stream is still running.  griddep_wait() blocks until that
// kernel has completed and its memory is visible (a no-op when the launch was
// ordinary); griddep_launch() lets the next kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA --------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y, int32_t z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Shared -> global 2-D tile store (TMA); elements outside the tensor are
// clipped.  Completion is tracked by bulk groups of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t x, int32_t y, const void *smem_src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(smem_src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load_1d(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- tcgen05 ----------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, f16 inputs, f32 accumulate.  A holds
// row i of the M x 16 slice in TMEM lane i, two f16 per 32-bit column in k
// order (lower half first), 8 columns from a_tmem.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with tf32 inputs taken from f32 operands in shared memory.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has
// completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns of TMEM into 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 registers per thread into 16 consecutive 32-bit TMEM columns of the
// thread's lane (32 lanes from taddr's lane field).
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 64 registers per thread into 64 consecutive 32-bit TMEM columns.
__device__ __forceinline__ void tmem_st_32x32b_x64(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row atoms of 1024 bytes (the stride
// byte offset), start address in 16-byte units, descriptor version 1,
// layout type 2 (SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);        // start address
    d |= (uint64_t)1u << 16;                             // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024u >> 4) << 32;                   // stride byte offset: next 8-row atom
    d |= (uint64_t)1u << 46;                             // descriptor version
    d |= (uint64_t)2u << 61;                             // SWIZZLE_128B
    return d;
}

// Instruction descriptor for kind::f16 / kind::tf32 with f32 accumulators,
// both operands K-major.  ab_format: 0 = f16, 2 = tf32.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t ab_format, uint32_t m, uint32_t n) {
    return (1u << 4)               // D format f32
           | (ab_format << 7)      // A format
           | (ab_format << 10)     // B format
           | ((n >> 3) << 17)      // N / 8
           | ((m >> 4) << 24);     // M / 16
}

// ---- thread-block clusters ----------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// (no memory clobber: the partials were published by the cluster barrier
// before the first of these loads and are not written again until the next one)
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
// (no memory clobber either: the flags it reads are written before the first
// cluster barrier; the loads may overlap the partial-tile loads that follow)
__device__ __forceinline__ int ld_dsmem_u32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// The end of a split-K epilogue: this CTA's reads of its peers' shared memory
// have returned (their values are in registers), so it arrives without
// release semantics -- the arrival does not wait for its own global stores to
// drain -- and then waits until every peer has done the same, so that no CTA
// leaves while another still reads its partial tile.
__device__ __forceinline__ void cluster_arrive_relaxed_wait() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// Butterfly reduction of V values (a power of two <= 32) over the warp:
// afterwards lane l holds the warp total of value l % V in a[0].
template <int V> __device__ __forceinline__ float warp_transpose_sum(float (&a)[V], int lane) {
#pragma unroll
    for (int h = V / 2; h >= 1; h >>= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int t = 0; t < h; ++t) {
            const float send = upper ? a[t] : a[t + h];
            const float keep = upper ? a[t + h] : a[t];
            a[t] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, h);
        }
    }
#pragma unroll
    for (int off = V; off < 32; off <<= 1) a[0] += __shfl_xor_sync(0xFFFFFFFFu, a[0], off);
    return a[0];
}

// Split-K epilogue of the tensor-core GEMMs: CTA z of a cluster of S sums
// column slice z (BN/S columns) of the S partial tiles, each [BN][ROWS] fp32
// at shared address red0 in every CTA of the cluster, in rank order 0..S-1,
// and stores it to dst[n][m] (row stride M).  Work items are 4 consecutive
// rows of one column, spread over nthreads threads; each thread keeps 16/S
// items' remote loads in flight before it sums any (a remote load costs
// hundreds of cycles).  skip: store nothing (a CTA of the cluster gave up);
// the loads still run, so they need not wait for the abort flags.
template <int S, int ROWS>
__device__ __forceinline__ void splitk_reduce_store_s(uint32_t red0, int z, int BN, int m0, int n0, int M, int N,
                                                      float *dst, int tid, int nthreads, bool skip) {
    constexpr int B = 16 / S;  // items in flight per thread
    const int cols = BN / S, c0 = z * cols;
    const int total = cols * (ROWS / 4);
    const bool vec = (M % 4) == 0;
    for (int it0 = tid; it0 < total; it0 += B * nthreads) {
        float4 v[B][S];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int it = it0 + u * nthreads;
            if (it < total) {
                const int cl = c0 + it / (ROWS / 4), r4 = (it % (ROWS / 4)) * 4;
                const uint32_t off = static_cast<uint32_t>((cl * ROWS + r4) * 4);
#pragma unroll
                for (int pr = 0; pr < S; ++pr) v[u][pr] = ld_dsmem_v4(mapa_shared(red0 + off, static_cast<uint32_t>(pr)));
            }
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int it = it0 + u * nthreads;
            if (it >= total) continue;
            const int cl = c0 + it / (ROWS / 4), r4 = (it % (ROWS / 4)) * 4;
            float4 acc = v[u][0];
#pragma unroll
            for (int pr = 1; pr < S; ++pr) {
                acc.x += v[u][pr].x;
                acc.y += v[u][pr].y;
                acc.z += v[u][pr].z;
                acc.w += v[u][pr].w;
            }
            const int gn = n0 + cl, gm = m0 + r4;
            if (!skip && gn < N && gm < M) {
                float *d = dst + static_cast<int64_t>(gn) * M + gm;
                if (vec && gm + 4 <= M) {
                    *reinterpret_cast<float4 *>(d) = acc;
                } else {
                    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
                    for (int t = 0; t < 4 && gm + t < M; ++t) d[t] = a4[t];
                }
            }
        }
    }
}

// The same for a runtime S in {2, 4, 8}.
template <int ROWS>
__device__ __forceinline__ void splitk_reduce_store(uint32_t red0, int S, int z, int BN, int m0, int n0, int M, int N,
                                                    float *dst, int tid, int nthreads, bool skip) {
    switch (S) {
    case 2: splitk_reduce_store_s<2, ROWS>(red0, z, BN, m0, n0, M, N, dst, tid, nthreads, skip); break;
    case 4: splitk_reduce_store_s<4, ROWS>(red0, z, BN, m0, n0, M, N, dst, tid, nthreads, skip); break;
    default: splitk_reduce_store_s<8, ROWS>(red0, z, BN, m0, n0, M, N, dst, tid, nthreads, skip); break;
    }
}

// Launch `kernel` on `st` with programmatic dependent launch allowed (and an
// optional cluster shape; 1 x 1 x 1 launches without clusters).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              dim3 cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster.x * cluster.y * cluster.z > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = cluster.x;
        attrs[na].val.clusterDim.y = cluster.y;
        attrs[na].val.clusterDim.z = cluster.z;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace qmm
