/*
 * synth.c -- seeded synthetic input generators shared by the tests, the
 * benchmark and the oracle checks.  Byte and float streams only: nothing here
 * decodes a format or computes a product.
 *
 *   synth_lcg_bytes   the 32-bit LCG byte stream of cera 0.4.0
 *                     examples/wgpu_gemm_bench.rs, fn fill_quant_bytes
 *                     (state = state*1664525 + 1013904223, byte = bits 16..23;
 *                     bit 6 cleared at odd offsets so f16 scales stay finite)
 *   synth_vecf        the xorshift64 float stream of memra-engine 0.128.0
 *                     src/bin/moe_rows_ceiling_bench.rs, fn vecf
 *                     (uniform in [-1, 1) with 24-bit resolution)
 *   synth_nvfp4_rows  the same page's fn synth_rows: per 36-byte group, four
 *                     scale bytes (r & 7) | 0x38, then 32 raw bytes, from an
 *                     LCG whose byte is the top 8 bits of the state
 */
#include <stdint.h>

void synth_lcg_bytes(uint32_t seed, uint8_t *out, int64_t len, int clear_bit6_odd) {
    uint32_t s = seed;
    for (int64_t i = 0; i < len; ++i) {
        s = s * 1664525u + 1013904223u;
        uint8_t b = (uint8_t)(s >> 16);
        if (clear_bit6_odd && (i & 1)) b &= 0xBF;
        out[i] = b;
    }
}

void synth_vecf(uint64_t seed, float *out, int64_t n) {
    uint64_t s = (seed * 0x9E3779B97F4A7C15ull) | 1ull;
    for (int64_t i = 0; i < n; ++i) {
        s ^= s << 13;
        s ^= s >> 7;
        s ^= s << 17;
        out[i] = ((float)(s >> 40) / 16777216.0f - 0.5f) * 2.0f;
    }
}

void synth_nvfp4_rows(uint32_t seed, uint8_t *out, int64_t groups) {
    uint32_t s = seed;
    for (int64_t g = 0; g < groups; ++g) {
        uint8_t *c = out + g * 36;
        for (int i = 0; i < 4; ++i) {
            s = s * 1664525u + 1013904223u;
            c[i] = (uint8_t)(((s >> 24) & 0x07u) | 0x38u);
        }
        for (int i = 4; i < 36; ++i) {
            s = s * 1664525u + 1013904223u;
            c[i] = (uint8_t)(s >> 24);
        }
    }
}
