// decode.cuh -- device decoders of the packed weight formats.
//
// Two forms:
//   Dec8<F, L>   8 consecutive weights of one block -> float32, each equal to
//                the format's value rounded once to float32 (bit-exact with
//                the definitions; used by the dequant kernel), read through a
//                global (LdG) or shared-memory (LdS) loader.
//   decode32_s<F> 32 consecutive weights staged in shared memory -> f16 in
//                k order (the A operand of the tensor-core GEMM).
//
// Block layouts (weights per block / bytes per block):
//   Q4_0 32/18: f16 d, 16 bytes; low nibble of byte j = element j, high
//               nibble = element j+16; value (q-8)*d.
//   Q8_0 32/34: f16 d, 32 int8; value q*d.
//   Q4_K 256/144: f16 d, f16 dmin, 12 bytes of 6-bit scales/mins, 128 bytes of
//               nibbles; element e: chunk c = e/64, r = e%64, byte 32c + r%32,
//               low nibble if r < 32; value d*sc*q - dmin*min (ggml k-quant
//               order).
//   Q6_K 256/210: 128 B low 4 bits, 64 B high 2 bits, 16 int8 scales, f16 d;
//               element e: h = e/128, r = e%128, s = r/32, l = r%32, low bits
//               in byte 64h + l + 32(s&1) (low nibble if s < 2), high bits
//               (qh[32h+l] >> 2s) & 3, scale 8h + l/16 + 2s; value
//               d*sc*(q-32).
//   NVFP4 64/36: 4 E4M3 scale bytes (one per 16), 32 bytes of E2M1 codes,
//               low nibble of byte j = element 2j; value e2m1*e4m3.
// (packed sizes: cera 0.4.0 examples/wgpu_gemm_bench.rs, VARIANTS; NVFP4:
// memra-engine 0.128.0 moe_rows_ceiling_bench.rs, synth_rows.)
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "common.cuh"

namespace qmm {

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// OCP E4M3FN byte -> float (exact; hardware conversion through f16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(hr));
}

// OCP E2M1 code (4 bits) -> float.  Twice the magnitudes {0,.5,1,1.5,2,3,4,6}
// are {0,1,2,3,4,6,8,12}, one nibble each of 0xC8643210.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
    const float mag = 0.5f * static_cast<float>((0xC8643210u >> (4u * (code & 7u))) & 15u);
    return (code & 8u) ? -mag : mag;
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

// Byte loaders: read-only global loads, or shared-memory loads through a
// generic pointer into shared memory.  The decoders below are written once
// against either.
struct LdG {
    static __device__ __forceinline__ uint32_t u8(const uint8_t *p) { return __ldg(p); }
    static __device__ __forceinline__ uint32_t u16(const uint8_t *p) {
        return __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    static __device__ __forceinline__ uint32_t u32(const uint8_t *p) {
        return __ldg(reinterpret_cast<const unsigned int *>(p));
    }
    static __device__ __forceinline__ uint2 u64(const uint8_t *p) { return __ldg(reinterpret_cast<const uint2 *>(p)); }
};
struct LdS {
    static __device__ __forceinline__ uint32_t u8(const uint8_t *p) {
        unsigned short v;
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
        return v;
    }
    static __device__ __forceinline__ uint32_t u16(const uint8_t *p) {
        unsigned short v;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
        return v;
    }
    static __device__ __forceinline__ uint32_t u32(const uint8_t *p) {
        uint32_t v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
        return v;
    }
    static __device__ __forceinline__ uint2 u64(const uint8_t *p) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
        return v;
    }
};
// 4 bytes from a 2-byte aligned address.
template <class L> __device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t *p) {
    return L::u16(p) | (L::u16(p + 2) << 16);
}

// Sub-block j (0..7) scale and min of a Q4_K superblock from its 12 scale bytes.
template <class L> __device__ __forceinline__ void q4k_sc_min(const uint8_t *sc12, int j, int &sc, int &mn) {
    if (j < 4) {
        sc = L::u8(sc12 + j) & 63;
        mn = L::u8(sc12 + j + 4) & 63;
    } else {
        const uint32_t b = L::u8(sc12 + j + 4);
        sc = static_cast<int>((b & 15u) | ((L::u8(sc12 + j - 4) >> 6) << 4));
        mn = static_cast<int>((b >> 4) | ((L::u8(sc12 + j) >> 6) << 4));
    }
}

// ---------------------------------------------------------------------------
// Dec8<F, L>::run: weights e..e+7 (e % 8 == 0) of the block at `blk`, as
// float32.  `ts` multiplies NVFP4 values after the exact e2m1*e4m3 product.
// ---------------------------------------------------------------------------
template <int F, class L> struct Dec8;

template <class L> struct Dec8<QMM_Q4_0, L> {
    static __device__ __forceinline__ void run(const uint8_t *blk, int e, float, float (&w)[8]) {
        const float d = half_bits_to_f32(L::u16(blk));
        const uint8_t *q = blk + 2 + (e & 15);
        const uint32_t lo = ld_u32_a2<L>(q), hi = ld_u32_a2<L>(q + 4);
        const int sh = (e >= 16) ? 4 : 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[j] = static_cast<float>(static_cast<int>((lo >> (8 * j + sh)) & 15u) - 8) * d;
            w[4 + j] = static_cast<float>(static_cast<int>((hi >> (8 * j + sh)) & 15u) - 8) * d;
        }
    }
};

template <class L> struct Dec8<QMM_Q8_0, L> {
    static __device__ __forceinline__ void run(const uint8_t *blk, int e, float, float (&w)[8]) {
        const float d = half_bits_to_f32(L::u16(blk));
        const uint8_t *q = blk + 2 + e;
        const uint32_t lo = ld_u32_a2<L>(q), hi = ld_u32_a2<L>(q + 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[j] = static_cast<float>(static_cast<int8_t>((lo >> (8 * j)) & 0xFFu)) * d;
            w[4 + j] = static_cast<float>(static_cast<int8_t>((hi >> (8 * j)) & 0xFFu)) * d;
        }
    }
};

template <class L> struct Dec8<QMM_Q4_K, L> {
    static __device__ __forceinline__ void run(const uint8_t *blk, int e, float, float (&w)[8]) {
        const uint32_t dd = L::u32(blk);
        const float d = half_bits_to_f32(dd & 0xFFFFu), dmin = half_bits_to_f32(dd >> 16);
        int sc, mn;
        q4k_sc_min<L>(blk + 4, e >> 5, sc, mn);
        const float a = __fmul_rn(d, static_cast<float>(sc));     // exact
        const float b = __fmul_rn(dmin, static_cast<float>(mn));  // exact
        const int c = e >> 6, r = e & 63;
        const uint2 q = L::u64(blk + 16 + 32 * c + (r & 31));
        const int sh = (r >= 32) ? 4 : 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[j] = __fmaf_rn(a, static_cast<float>((q.x >> (8 * j + sh)) & 15u), -b);
            w[4 + j] = __fmaf_rn(a, static_cast<float>((q.y >> (8 * j + sh)) & 15u), -b);
        }
    }
};

template <class L> struct Dec8<QMM_Q6_K, L> {
    static __device__ __forceinline__ void run(const uint8_t *blk, int e, float, float (&w)[8]) {
        const int h = e >> 7, r = e & 127, s = r >> 5, l = r & 31;
        const float d = half_bits_to_f32(L::u16(blk + 208));
        const int sc = static_cast<int8_t>(L::u8(blk + 192 + 8 * h + (l >> 4) + 2 * s));
        const float a = __fmul_rn(d, static_cast<float>(sc));  // exact
        const uint8_t *ql = blk + 64 * h + l + 32 * (s & 1);
        const uint8_t *qh = blk + 128 + 32 * h + l;
        const uint32_t ql0 = ld_u32_a2<L>(ql), ql1 = ld_u32_a2<L>(ql + 4);
        const uint32_t qh0 = ld_u32_a2<L>(qh), qh1 = ld_u32_a2<L>(qh + 4);
        const int lsh = (s >= 2) ? 4 : 0, hsh = 2 * s;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q0 = static_cast<int>(((ql0 >> (8 * j + lsh)) & 15u) | (((qh0 >> (8 * j + hsh)) & 3u) << 4));
            const int q1 = static_cast<int>(((ql1 >> (8 * j + lsh)) & 15u) | (((qh1 >> (8 * j + hsh)) & 3u) << 4));
            w[j] = __fmul_rn(a, static_cast<float>(q0 - 32));  // exact
            w[4 + j] = __fmul_rn(a, static_cast<float>(q1 - 32));
        }
    }
};

template <class L> struct Dec8<QMM_NVFP4, L> {
    static __device__ __forceinline__ void run(const uint8_t *blk, int e, float ts, float (&w)[8]) {
        const float s = e4m3_to_f32(L::u8(blk + (e >> 4)));
        const uint32_t codes = L::u32(blk + 4 + (e >> 1));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float v = __fmul_rn(e2m1_to_f32((codes >> (4 * j)) & 15u), s);  // exact
            w[j] = __fmul_rn(v, ts);
        }
    }
};

// f32 weights: 8 consecutive weights of a row from element e (bounds-checked
// against k); `row` points at the row's first weight.
template <class L> __device__ __forceinline__ void decode8_f32(const uint8_t *row, int64_t e, int64_t k, float (&w)[8]) {
    const uint8_t *p = row + 4 * e;
    if (e + 8 <= k && (reinterpret_cast<uintptr_t>(p) & 7u) == 0) {
        const uint2 a = L::u64(p), b = L::u64(p + 8), c = L::u64(p + 16), d = L::u64(p + 24);
        w[0] = __uint_as_float(a.x); w[1] = __uint_as_float(a.y); w[2] = __uint_as_float(b.x); w[3] = __uint_as_float(b.y);
        w[4] = __uint_as_float(c.x); w[5] = __uint_as_float(c.y); w[6] = __uint_as_float(d.x); w[7] = __uint_as_float(d.y);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = (e + j < k) ? __uint_as_float(L::u32(p + 4 * j)) : 0.0f;
    }
}

// ---------------------------------------------------------------------------
// decode32_s: weights e0..e0+31 (e0 % 32 == 0) of a raw weight segment staged
// in shared memory, as 16 half2 words in k order (the A operand of the
// tensor-core GEMM).  `a` is the shared-memory address of the segment's first
// block (2-byte aligned); e0 counts from that block.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }
__device__ __forceinline__ __half2 bits_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
// N little-endian words starting at any 2-byte aligned shared address:
// aligned loads, then a funnel shift by the byte offset.
template <int N> __device__ __forceinline__ void lds_words(uint32_t a, uint32_t (&out)[N]) {
    const uint32_t base = a & ~3u, sh = (a & 3u) * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = lds_u32(base + 4u * i);
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

template <int F> __device__ __forceinline__ void decode32_s(uint32_t a, int e0, uint32_t (&o)[16]);

// Q4_0: one whole block.  (1024 + q) is built by OR-ing the nibble into the
// f16 pattern of 1024.0; subtracting 1032 gives q - 8 exactly; one multiply by
// d rounds once (round to nearest even).
template <> __device__ __forceinline__ void decode32_s<QMM_Q4_0>(uint32_t a, int e0, uint32_t (&o)[16]) {
    const uint32_t blk = a + 18u * static_cast<uint32_t>(e0 >> 5);
    const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(lds_u16(blk))));
    const __half2 off = __floats2half2_rn(1032.0f, 1032.0f);
    uint32_t q[4];
    lds_words<4>(blk + 2, q);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t v = q[t], vh = v >> 4;
        // elements 4t..4t+3 (low nibbles) and 16+4t..16+4t+3 (high nibbles)
        const uint32_t l01 = (__byte_perm(v, 0, 0x4140) & 0x000F000Fu) | 0x64006400u;
        const uint32_t l23 = (__byte_perm(v, 0, 0x4342) & 0x000F000Fu) | 0x64006400u;
        const uint32_t h01 = (__byte_perm(vh, 0, 0x4140) & 0x000F000Fu) | 0x64006400u;
        const uint32_t h23 = (__byte_perm(vh, 0, 0x4342) & 0x000F000Fu) | 0x64006400u;
        o[2 * t] = h2_bits(__hmul2(__hsub2(bits_h2(l01), off), d2));
        o[2 * t + 1] = h2_bits(__hmul2(__hsub2(bits_h2(l23), off), d2));
        o[8 + 2 * t] = h2_bits(__hmul2(__hsub2(bits_h2(h01), off), d2));
        o[8 + 2 * t + 1] = h2_bits(__hmul2(__hsub2(bits_h2(h23), off), d2));
    }
}

// Q8_0: one whole block.  Flipping the sign bit gives q + 128 as an unsigned
// byte; placed under the f16 exponent of 1024 it reads 1024 + q + 128, minus
// 1152 is q exactly; one multiply by d rounds once.
template <> __device__ __forceinline__ void decode32_s<QMM_Q8_0>(uint32_t a, int e0, uint32_t (&o)[16]) {
    const uint32_t blk = a + 34u * static_cast<uint32_t>(e0 >> 5);
    const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(lds_u16(blk))));
    const __half2 off = __floats2half2_rn(1152.0f, 1152.0f);
    uint32_t q[8];
    lds_words<8>(blk + 2, q);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t v = q[t] ^ 0x80808080u;
        o[2 * t] = h2_bits(__hmul2(__hsub2(bits_h2(__byte_perm(v, 0x64646464u, 0x4140)), off), d2));
        o[2 * t + 1] = h2_bits(__hmul2(__hsub2(bits_h2(__byte_perm(v, 0x64646464u, 0x4342)), off), d2));
    }
}

// Byte i (0..11, warp-uniform) of the Q4_K scale area held in three words.
__device__ __forceinline__ uint32_t sc12_byte(uint32_t w0, uint32_t w1, uint32_t w2, int i) {
    const uint32_t w = i < 4 ? w0 : (i < 8 ? w1 : w2);
    return (w >> (8 * (i & 3))) & 0xFFu;
}

// Q4_K: one 32-weight sub-block of the superblock at `a` (16-byte aligned),
// computed in float32 as one fused d*sc*q - dmin*min (both products exact),
// then rounded to f16.
template <> __device__ __forceinline__ void decode32_s<QMM_Q4_K>(uint32_t a, int e0, uint32_t (&o)[16]) {
    const uint4 hd = lds_v4(a);
    const float d = half_bits_to_f32(hd.x & 0xFFFFu), dmin = half_bits_to_f32(hd.x >> 16);
    const int j = e0 >> 5;
    uint32_t sc, mn;
    if (j < 4) {
        sc = sc12_byte(hd.y, hd.z, hd.w, j) & 63u;
        mn = sc12_byte(hd.y, hd.z, hd.w, j + 4) & 63u;
    } else {
        const uint32_t b = sc12_byte(hd.y, hd.z, hd.w, j + 4);
        sc = (b & 15u) | ((sc12_byte(hd.y, hd.z, hd.w, j - 4) >> 6) << 4);
        mn = (b >> 4) | ((sc12_byte(hd.y, hd.z, hd.w, j) >> 6) << 4);
    }
    const float av = __fmul_rn(d, static_cast<float>(sc));
    const float bv = __fmul_rn(dmin, static_cast<float>(mn));
    const int sh = (e0 & 32) ? 4 : 0;
    const uint32_t qa = a + 16u + 32u * static_cast<uint32_t>(e0 >> 6);
    const uint4 q0 = lds_v4(qa), q1 = lds_v4(qa + 16u);
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t v = words[t] >> sh;
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __fmaf_rn(av, static_cast<float>((v >> (8 * i)) & 15u), -bv);
        o[2 * t] = h2_bits(__floats2half2_rn(f[0], f[1]));
        o[2 * t + 1] = h2_bits(__floats2half2_rn(f[2], f[3]));
    }
}

// Q6_K: one 32-weight quadrant (h, s) of the superblock at `a`;
// (d*sc)*(q-32) is exact in float32, so the conversion to f16 is the only
// rounding.
template <> __device__ __forceinline__ void decode32_s<QMM_Q6_K>(uint32_t a, int e0, uint32_t (&o)[16]) {
    const int h = e0 >> 7, s = (e0 >> 5) & 3;
    const float d = half_bits_to_f32(lds_u16(a + 208u));
    const uint32_t sc2 = lds_u16(a + 192u + 8u * h + 2u * s);
    const float a0 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(sc2 & 0xFFu)));
    const float a1 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(sc2 >> 8)));
    uint32_t ql[8], qh[8];
    lds_words<8>(a + 64u * h + 32u * (s & 1), ql);
    lds_words<8>(a + 128u + 32u * h, qh);
    const int lsh = (s >= 2) ? 4 : 0, hsh = 2 * s;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t q = ((ql[t] >> lsh) & 0x0F0F0F0Fu) | (((qh[t] >> hsh) & 0x03030303u) << 4);
        const float av = (t < 4) ? a0 : a1;
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __fmul_rn(av, static_cast<float>(static_cast<int>((q >> (8 * i)) & 63u) - 32));
        o[2 * t] = h2_bits(__floats2half2_rn(f[0], f[1]));
        o[2 * t + 1] = h2_bits(__floats2half2_rn(f[2], f[3]));
    }
}

// NVFP4: half of the 64-weight group at a + 36*(e0/64) (4-byte aligned);
// e2m1*e4m3 has at most 6 significant bits and lies in [2^-10, 2688], so the
// f16 product is exact.
template <> __device__ __forceinline__ void decode32_s<QMM_NVFP4>(uint32_t a, int e0, uint32_t (&o)[16]) {
    const uint32_t grp = a + 36u * static_cast<uint32_t>(e0 >> 6);
    const uint32_t hf = static_cast<uint32_t>((e0 >> 5) & 1);
    const uint32_t sc2 = lds_u16(grp + 2u * hf);
    const __half2 s0 = __float2half2_rn(e4m3_to_f32(sc2 & 0xFFu));
    const __half2 s1 = __float2half2_rn(e4m3_to_f32(sc2 >> 8));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t c = lds_u32(grp + 4u + 16u * hf + 4u * t);
        const __half2 sv = (t < 2) ? s0 : s1;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t byte = (c >> (8 * i)) & 0xFFu;
            const __half2 v = __floats2half2_rn(e2m1_to_f32(byte & 15u), e2m1_to_f32(byte >> 4));
            o[4 * t + i] = h2_bits(__hmul2(v, sv));
        }
    }
}

// ---------------------------------------------------------------------------
// dec128_aligned<F, H>: weights 128H .. 128H+127 of a 256-wide raw segment
// whose first byte is 16-byte aligned in shared memory (row bytes a multiple
// of 16), as 64 half2 words in k order.  The segment bytes come in with
// 16-byte loads -- conflict-free across a warp's 32 rows because the row pitch
// is an odd multiple of 16 bytes -- and every block sits at a compile-time
// byte offset, so the extraction is static funnel shifts.  Results are the
// same bits as decode32_s.
// ---------------------------------------------------------------------------
template <int NW> __device__ __forceinline__ uint32_t word_at(const uint32_t (&w)[NW], int b) {
    const int i = b >> 2, sh = (b & 3) * 8;
    return sh == 0 ? w[i] : __funnelshift_r(w[i], w[i + 1], sh);
}
template <int NCH, int NW> __device__ __forceinline__ void lds_chunks(uint32_t a, uint32_t (&w)[NW]) {
    static_assert(NW >= 4 * NCH + 1, "one spare word");
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const uint4 v = lds_v4(a + 16u * i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    w[4 * NCH] = 0u;
}

template <int F, int H> struct Dec128 {  // formats without an aligned variant: never called
    static __device__ __forceinline__ void run(uint32_t, uint32_t (&o)[64]) {
#pragma unroll
        for (int i = 0; i < 64; ++i) o[i] = 0u;
    }
};

template <int H> struct Dec128<QMM_Q4_0, H> {
    static __device__ __forceinline__ void run(uint32_t a, uint32_t (&o)[64]) {
        constexpr int LO = H ? 64 : 0, OFF = 72 * H - LO;  // 4 blocks of 18 bytes from byte 72H
        uint32_t w[21];
        lds_chunks<5>(a + LO, w);
        const __half2 off = __floats2half2_rn(1032.0f, 1032.0f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = OFF + 18 * j;
            const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(word_at(w, b) & 0xFFFFu)));
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t v = word_at(w, b + 2 + 4 * t), vh = v >> 4;
                const uint32_t l01 = (__byte_perm(v, 0, 0x4140) & 0x000F000Fu) | 0x64006400u;
                const uint32_t l23 = (__byte_perm(v, 0, 0x4342) & 0x000F000Fu) | 0x64006400u;
                const uint32_t h01 = (__byte_perm(vh, 0, 0x4140) & 0x000F000Fu) | 0x64006400u;
                const uint32_t h23 = (__byte_perm(vh, 0, 0x4342) & 0x000F000Fu) | 0x64006400u;
                o[16 * j + 2 * t] = h2_bits(__hmul2(__hsub2(bits_h2(l01), off), d2));
                o[16 * j + 2 * t + 1] = h2_bits(__hmul2(__hsub2(bits_h2(l23), off), d2));
                o[16 * j + 8 + 2 * t] = h2_bits(__hmul2(__hsub2(bits_h2(h01), off), d2));
                o[16 * j + 8 + 2 * t + 1] = h2_bits(__hmul2(__hsub2(bits_h2(h23), off), d2));
            }
        }
    }
};

template <int H> struct Dec128<QMM_Q8_0, H> {
    static __device__ __forceinline__ void run(uint32_t a, uint32_t (&o)[64]) {
        constexpr int LO = H ? 128 : 0, OFF = 136 * H - LO;  // 4 blocks of 34 bytes from byte 136H
        uint32_t w[37];
        lds_chunks<9>(a + LO, w);
        const __half2 off = __floats2half2_rn(1152.0f, 1152.0f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = OFF + 34 * j;
            const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(word_at(w, b) & 0xFFFFu)));
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t v = word_at(w, b + 2 + 4 * t) ^ 0x80808080u;
                o[16 * j + 2 * t] = h2_bits(__hmul2(__hsub2(bits_h2(__byte_perm(v, 0x64646464u, 0x4140)), off), d2));
                o[16 * j + 2 * t + 1] =
                    h2_bits(__hmul2(__hsub2(bits_h2(__byte_perm(v, 0x64646464u, 0x4342)), off), d2));
            }
        }
    }
};

template <int H> struct Dec128<QMM_NVFP4, H> {
    static __device__ __forceinline__ void run(uint32_t a, uint32_t (&o)[64]) {
        constexpr int LO = H ? 64 : 0, OFF = 72 * H - LO;  // 2 groups of 36 bytes from byte 72H
        uint32_t w[21];
        lds_chunks<5>(a + LO, w);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int b = OFF + 36 * g;
            const uint32_t sc4 = word_at(w, b);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const __half2 s0 = __float2half2_rn(e4m3_to_f32((sc4 >> (16 * hf)) & 0xFFu));
                const __half2 s1 = __float2half2_rn(e4m3_to_f32((sc4 >> (16 * hf + 8)) & 0xFFu));
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t c = word_at(w, b + 4 + 16 * hf + 4 * t);
                    const __half2 sv = (t < 2) ? s0 : s1;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t byte = (c >> (8 * i)) & 0xFFu;
                        const __half2 v = __floats2half2_rn(e2m1_to_f32(byte & 15u), e2m1_to_f32(byte >> 4));
                        o[32 * g + 16 * hf + 4 * t + i] = h2_bits(__hmul2(v, sv));
                    }
                }
            }
        }
    }
};

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

// NVFP4 V2 row (k/2 code bytes, then k/16 E4M3 scale bytes): the same
// decode as the 36-byte groups, with the codes at e0/2 and the scale at
// k/2 + e0/16 (k % 64 == 0 keeps the code word 4-byte aligned).
template <> __device__ __forceinline__ void grp8<QMM_NVFP4_V2>(const uint8_t *row, int64_t e0, int64_t k, Grp &g) {
    g.scale = 0.5f * e4m3_to_f32(LdS::u8(row + (k >> 1) + (e0 >> 4)));  // the bytes below hold 2 * value
    g.offset = 0.0f;
    const uint32_t codes = LdS::u32(row + (e0 >> 1));
    const uint32_t lo = e2m1x4_offset_bytes(codes & 0xFFFFu), hi = e2m1x4_offset_bytes(codes >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g.v[j] = byte_as_float(lo, j, 8388620.0f);  // (2v + 12) - 12
        g.v[4 + j] = byte_as_float(hi, j, 8388620.0f);
    }
}

// Packed pairs of f32 (Blackwell f32x2 arithmetic: two independent
// round-to-nearest operations per instruction, same results as scalar ones).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Two E2M1 codes of one byte as an exact f32 pair (element of the low nibble
// first): the hardware E2M1 -> f16x2 conversion, then f16 -> f32 widening,
// both exact for every code.
__device__ __forceinline__ uint64_t f16x2_to_f2(uint32_t h) {
    uint64_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 a, b;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.f32.f16 a, lo;\n\t"
        "cvt.f32.f16 b, hi;\n\t"
        "mov.b64 %0, {a, b};\n\t}"
        : "=l"(r) : "r"(h));
    return r;
}
__device__ __forceinline__ void e2m1x8_to_f2(uint32_t c, uint64_t *w) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(c));
    w[0] = f16x2_to_f2(h0);
    w[1] = f16x2_to_f2(h1);
    w[2] = f16x2_to_f2(h2);
    w[3] = f16x2_to_f2(h3);
}

}  // namespace qmm
