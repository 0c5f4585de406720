/*
 * qmm_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * quantized-weight projection matmul dst[n][m] = sum_k W[m][k] * X[n][k].
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and may
 * be loaded only by tests/, by __graft_entry__.smoke() and by bench.py's
 * cpu_baseline / --impl reference leg.  It shares no code, header, table or
 * constant with the CUDA library under gemv_dequant_gemm_gb300/, and that
 * library never calls it.
 *
 * Every value is decoded to double precision from the formats' definitions and
 * every sum is a plain double loop in k order.  No blocking, no fusion, no
 * reordering.  Citations name the page and the item on it:
 *
 *   [cera]   cera 0.4.0, examples/wgpu_gemm_bench.rs
 *              - doc comment of struct Shape: the benchmarked product takes
 *                src0 [m][k] and src1 [n][k] to dst [n][m]
 *              - VARIANTS table: packed sizes 4 B/weight (f32), 18 B/32
 *                (q4_0), 34 B/32 (q8_0), 144 B/256 (q4_k), 210 B/256 (q6_k)
 *              - fill_quant_bytes doc comment: every f16 scale sits at an even
 *                offset with its high byte at an odd offset
 *              - comparison comment in main: dst rows have stride m
 *   [memra]  memra-engine 0.128.0, src/bin/moe_rows_ceiling_bench.rs
 *              - synth_rows: NVFP4 row = in_f/64 groups of 36 B, 4 E4M3 scale
 *                bytes then 32 B of E2M1 nibbles
 *              - main: pointer table index plane*n_pairs + j, per-matrix scale
 *                scl[pr] = 0.5 + 0.01*pr, gate = plane 0, up = plane 1
 *              - main, the V2 arms: the same values repacked "split" so that
 *                each row holds 18 B per 32 weights (16 B of codes, 2 scale
 *                bytes) with the scales as one contiguous stream
 *   [hrx]    hrx-rs patch_bench.rs, fn float: the binary16 decode with
 *              subnormals (exponent field 0 -> mantissa * 2^-24)
 *   [aprender] aprender-serve 0.70.2 cublas_prefill/mod.rs, module doc: its
 *              v1 prefill path dequantizes weights to FP32 first (the
 *              standalone dequant step)
 *
 * Readings where the pages are silent (the byte orderings inside Q4_K and
 * Q6_K, the NVFP4 nibble order, the MoE output layout, the V2 row layout, the
 * Q8_1 block rule) follow the workload definitions stated alongside the
 * benchmark; each is stated at the function that takes it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Format codes of this oracle (its own numbering). */
enum {
    ORC_F32 = 0,
    ORC_Q4_0 = 1,
    ORC_Q8_0 = 2,
    ORC_Q4_K = 3,
    ORC_Q6_K = 4,
    ORC_NVFP4 = 5,
    ORC_NVFP4_V2 = 6
};

/* ---------------------------------------------------------------------- */
/* Scalar codes                                                             */
/* ---------------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Exponent field 0 is a subnormal mantissa * 2^-24 ([hrx] fn float), 31 is
 * Inf (fraction 0) or NaN. */
double oracle_fp16(uint32_t code) {
    uint32_t sign = (code >> 15) & 1u;
    uint32_t expo = (code >> 10) & 31u;
    uint32_t frac = code & 1023u;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = frac == 0 ? INFINITY : NAN;
    } else {
        mag = ldexp(1.0 + (double)frac / 1024.0, (int)expo - 15);
    }
    return sign ? -mag : mag;
}

/* OCP FP8 E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (mantissa/8 * 2^-6); S.1111.111 is NaN; there
 * is no infinity.  [memra] synth_rows writes the scale bytes (r & 7) | 0x38. */
double oracle_e4m3(uint32_t code) {
    uint32_t sign = (code >> 7) & 1u;
    uint32_t expo = (code >> 3) & 15u;
    uint32_t mant = code & 7u;
    double mag;
    if (expo == 15 && mant == 7) {
        mag = NAN;
    } else if (expo == 0) {
        mag = ldexp((double)mant / 8.0, -6);
    } else {
        mag = ldexp(1.0 + (double)mant / 8.0, (int)expo - 7);
    }
    return sign ? -mag : mag;
}

/* OCP FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Exponent field 0 is subnormal (mantissa/2). */
double oracle_e2m1(uint32_t nibble) {
    uint32_t sign = (nibble >> 3) & 1u;
    uint32_t expo = (nibble >> 1) & 3u;
    uint32_t mant = nibble & 1u;
    double mag;
    if (expo == 0) {
        mag = (double)mant / 2.0;
    } else {
        mag = ldexp(1.0 + (double)mant / 2.0, (int)expo - 1);
    }
    return sign ? -mag : mag;
}

/* ---------------------------------------------------------------------- */
/* Block formats                                                            */
/* ---------------------------------------------------------------------- */

/* Weights per block ([cera] VARIANTS; [memra] synth_rows uses 64). */
int64_t oracle_block_weights(int fmt) {
    switch (fmt) {
    case ORC_F32: return 1;
    case ORC_Q4_0: return 32;
    case ORC_Q8_0: return 32;
    case ORC_Q4_K: return 256;
    case ORC_Q6_K: return 256;
    case ORC_NVFP4: return 64;
    case ORC_NVFP4_V2: return 32;
    default: return 0;
    }
}

/* Bytes per block ([cera] VARIANTS src0_bytes; [memra] 36 B per 64). */
int64_t oracle_block_bytes(int fmt) {
    switch (fmt) {
    case ORC_F32: return 4;
    case ORC_Q4_0: return 18;
    case ORC_Q8_0: return 34;
    case ORC_Q4_K: return 144;
    case ORC_Q6_K: return 210;
    case ORC_NVFP4: return 36;
    case ORC_NVFP4_V2: return 18;
    default: return 0;
    }
}

static double half_at(const uint8_t *p) {
    return oracle_fp16((uint32_t)p[0] | ((uint32_t)p[1] << 8));
}

/* Q4_0, 18 bytes: f16 d, then 16 bytes; the low nibble of byte j is element
 * j, the high nibble is element j+16; value (q - 8) * d. */
static void decode_q4_0(const uint8_t *b, double *out) {
    double d = half_at(b);
    for (int j = 0; j < 16; ++j) {
        int lo = b[2 + j] & 15;
        int hi = b[2 + j] >> 4;
        out[j] = (double)(lo - 8) * d;
        out[j + 16] = (double)(hi - 8) * d;
    }
}

/* Q8_0, 34 bytes: f16 d, then 32 signed bytes; value q * d. */
static void decode_q8_0(const uint8_t *b, double *out) {
    double d = half_at(b);
    for (int j = 0; j < 32; ++j) {
        int q = (int)(int8_t)b[2 + j];
        out[j] = (double)q * d;
    }
}

/* The 6-bit scale and min of sub-block j (0..7) of a Q4_K superblock, packed
 * in 12 bytes: sub-blocks 0..3 keep theirs in the low 6 bits of bytes j and
 * j+4; sub-blocks 4..7 take their low 4 bits from byte j+4 (scale: low
 * nibble, min: high nibble) and their high 2 bits from the top bits of bytes
 * j-4 (scale) and j (min). */
static void q4k_scale_min(const uint8_t *sc12, int j, int *sc, int *mn) {
    if (j < 4) {
        *sc = sc12[j] & 63;
        *mn = sc12[j + 4] & 63;
    } else {
        *sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
        *mn = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
}

/* Q4_K, 144 bytes: f16 d, f16 dmin, 12 bytes of scales/mins, 128 bytes of
 * nibbles.  Element e lies in 64-element chunk c = e/64; with r = e%64 its
 * nibble is byte 32c + r%32 of the nibble area, low for r < 32 and high
 * otherwise; it belongs to sub-block e/32.  Value d*sc*q - dmin*min. */
static void decode_q4_k(const uint8_t *b, double *out) {
    double d = half_at(b);
    double dmin = half_at(b + 2);
    const uint8_t *sc12 = b + 4;
    const uint8_t *qs = b + 16;
    for (int e = 0; e < 256; ++e) {
        int c = e / 64, r = e % 64;
        uint8_t byte = qs[32 * c + r % 32];
        int q = r < 32 ? (byte & 15) : (byte >> 4);
        int sc, mn;
        q4k_scale_min(sc12, e / 32, &sc, &mn);
        out[e] = d * (double)sc * (double)q - dmin * (double)mn;
    }
}

/* Q6_K, 210 bytes: 128 bytes of low 4 bits, 64 bytes of high 2 bits, 16
 * signed sub-block scales (16 weights each), f16 d.  Element e lies in half
 * h = e/128; with r = e%128, quadrant s = r/32 and l = r%32 its low 4 bits are
 * the low (s < 2) or high (s >= 2) nibble of byte 64h + l + 32*(s&1), its high
 * 2 bits are bits 2s..2s+1 of byte 32h + l of the high area, and its scale is
 * number 8h + l/16 + 2s.  Value d * sc * (q - 32). */
static void decode_q6_k(const uint8_t *b, double *out) {
    const uint8_t *ql = b;
    const uint8_t *qh = b + 128;
    const int8_t *scales = (const int8_t *)(b + 192);
    double d = half_at(b + 208);
    for (int e = 0; e < 256; ++e) {
        int h = e / 128, r = e % 128, s = r / 32, l = r % 32;
        uint8_t lowbyte = ql[64 * h + l + 32 * (s & 1)];
        int low = s < 2 ? (lowbyte & 15) : (lowbyte >> 4);
        int high = (qh[32 * h + l] >> (2 * s)) & 3;
        int q = low | (high << 4);
        int sc = scales[8 * h + l / 16 + 2 * s];
        out[e] = d * (double)sc * (double)(q - 32);
    }
}

/* NVFP4 group, 36 bytes ([memra] synth_rows): 4 E4M3 scale bytes, byte i
 * covering elements 16i..16i+15, then 32 bytes of E2M1 codes; the low nibble of
 * byte j is element 2j and the high nibble element 2j+1.  Value e2m1 * e4m3. */
static void decode_nvfp4(const uint8_t *b, double *out) {
    for (int e = 0; e < 64; ++e) {
        uint8_t byte = b[4 + e / 2];
        uint32_t nib = (e % 2 == 0) ? (byte & 15u) : (byte >> 4);
        out[e] = oracle_e2m1(nib) * oracle_e4m3(b[e / 16]);
    }
}

/* NVFP4 V2 row of k weights ([memra] main, the V2 arms; the byte order is
 * the reading that keeps each 32-weight code group on a 16-byte boundary):
 * first the k/2 code bytes (the low nibble of byte j is element 2j, the high
 * nibble element 2j+1, as in the 36-byte groups), then the k/16 E4M3 scale
 * bytes, scale byte s covering elements 16s..16s+15.  Value e2m1 * e4m3. */
static void decode_nvfp4_v2_row(const uint8_t *row, int64_t k, double *out) {
    const uint8_t *scales = row + k / 2;
    for (int64_t e = 0; e < k; ++e) {
        uint8_t byte = row[e / 2];
        uint32_t nib = (e % 2 == 0) ? (byte & 15u) : (byte >> 4);
        out[e] = oracle_e2m1(nib) * oracle_e4m3(scales[e / 16]);
    }
}

/* Decode one packed row of k weights into out[0..k).  Returns 0, or -1 for an
 * unknown format or a k that is not a whole number of blocks. */
int oracle_decode_row(int fmt, const uint8_t *row, int64_t k, double *out) {
    int64_t qk = oracle_block_weights(fmt);
    int64_t bb = oracle_block_bytes(fmt);
    if (qk == 0 || k < 0 || k % qk != 0) return -1;
    if (fmt == ORC_NVFP4_V2) {
        decode_nvfp4_v2_row(row, k, out);
        return 0;
    }
    for (int64_t blk = 0; blk < k / qk; ++blk) {
        const uint8_t *b = row + blk * bb;
        double *o = out + blk * qk;
        switch (fmt) {
        case ORC_F32: {
            float f;
            memcpy(&f, b, 4);
            o[0] = (double)f;
            break;
        }
        case ORC_Q4_0: decode_q4_0(b, o); break;
        case ORC_Q8_0: decode_q8_0(b, o); break;
        case ORC_Q4_K: decode_q4_k(b, o); break;
        case ORC_Q6_K: decode_q6_k(b, o); break;
        case ORC_NVFP4: decode_nvfp4(b, o); break;
        default: return -1;
        }
    }
    return 0;
}

/* Row stride in bytes of a packed [m][k] matrix: k / QK * block bytes. */
int64_t oracle_row_bytes(int fmt, int64_t k) {
    int64_t qk = oracle_block_weights(fmt);
    if (qk == 0 || k % qk != 0) return 0;
    return k / qk * oracle_block_bytes(fmt);
}

/* ---------------------------------------------------------------------- */
/* NVFP4 36-byte groups -> V2 rows ([memra] main: the V2 arms read the same    */
/* values, repacked)                                                        */
/* ---------------------------------------------------------------------- */

/* v2[m][k/32*18] from v1[m][k/64*36]: for every row, group g's 32 code bytes
 * go to bytes 32g..32g+31 of the row's code area and its 4 scale bytes to
 * bytes 4g..4g+3 of the scale area that follows (at k/2).  Returns -1 unless
 * k is a positive multiple of 64. */
int oracle_nvfp4_repack_v2(const uint8_t *v1, uint8_t *v2, int64_t m, int64_t k) {
    if (k <= 0 || k % 64 != 0 || m < 0) return -1;
    int64_t rb1 = k / 64 * 36, rb2 = k / 32 * 18;
    for (int64_t r = 0; r < m; ++r) {
        const uint8_t *src = v1 + r * rb1;
        uint8_t *dst = v2 + r * rb2;
        for (int64_t g = 0; g < k / 64; ++g) {
            for (int j = 0; j < 32; ++j) dst[32 * g + j] = src[36 * g + 4 + j];
            for (int j = 0; j < 4; ++j) dst[k / 2 + 4 * g + j] = src[36 * g + j];
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Standalone dequant ([aprender] v1 path: packed weights -> FP32)          */
/* ---------------------------------------------------------------------- */

/* out[m][k] = (float)(decoded value * tensor_scale).  Every decoded value is
 * exact in double and the product with a float tensor_scale has at most 30
 * significant bits, so the one rounding is the conversion to float. */
int oracle_dequant(int fmt, const uint8_t *w, int64_t m, int64_t k, double tensor_scale,
                   float *out) {
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    if (!tmp) return -2;
    for (int64_t r = 0; r < m; ++r) {
        if (oracle_decode_row(fmt, w + r * rb, k, tmp) != 0) {
            free(tmp);
            return -1;
        }
        for (int64_t c = 0; c < k; ++c) {
            double v = tmp[c];
            if (fmt == ORC_NVFP4 || fmt == ORC_NVFP4_V2) v = v * tensor_scale;
            out[r * k + c] = (float)v;
        }
    }
    free(tmp);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* The product ([cera] struct Shape doc comment)                            */
/* ---------------------------------------------------------------------- */

/* dst[i][j] = sum_c W[j][c] * X[i][c] and absmag[i][j] = sum_c |W[j][c]*X[i][c]|
 * for i < n, j < m, both [n][m] with row stride m.  X is [n][k] with row
 * stride k.  W rows are decoded once into a double matrix first. */
int oracle_matmul(int fmt, const uint8_t *w, const float *x, int64_t m, int64_t k, int64_t n,
                  double *dst, double *absmag, int threads) {
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(m * k > 0 ? m * k : 1));
    if (!wd) return -2;
    int bad = 0;
    for (int64_t r = 0; r < m; ++r)
        if (oracle_decode_row(fmt, w + r * rb, k, wd + r * k) != 0) bad = 1;
    if (bad) {
        free(wd);
        return -1;
    }
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t idx = 0; idx < n * m; ++idx) {
        int64_t i = idx / m, j = idx % m;
        double s = 0.0, a = 0.0;
        for (int64_t c = 0; c < k; ++c) {
            double p = wd[j * k + c] * (double)x[i * k + c];
            s += p;
            a += fabs(p);
        }
        dst[idx] = s;
        if (absmag) absmag[idx] = a;
    }
    free(wd);
    (void)threads;
    return 0;
}

/* The same sums for `count` chosen entries (ni[e], mj[e]) only, decoding just
 * the rows they need: the check for shapes too large to compute whole. */
int oracle_matmul_entries(int fmt, const uint8_t *w, const float *x, int64_t m, int64_t k,
                          int64_t n, int64_t count, const int64_t *ni, const int64_t *mj,
                          double *dst, double *absmag, int threads) {
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t e = 0; e < count; ++e) {
        int64_t i = ni[e], j = mj[e];
        if (i < 0 || i >= n || j < 0 || j >= m) {
            bad |= 1;
            continue;
        }
        double *row = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
        if (!row || oracle_decode_row(fmt, w + j * rb, k, row) != 0) {
            bad |= 1;
            free(row);
            continue;
        }
        double s = 0.0, a = 0.0;
        for (int64_t c = 0; c < k; ++c) {
            double p = row[c] * (double)x[i * k + c];
            s += p;
            a += fabs(p);
        }
        dst[e] = s;
        if (absmag) absmag[e] = a;
        free(row);
    }
    (void)threads;
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------- */
/* MoE gate/up GEMV ([memra] main: served kernel over the pointer table)   */
/* ---------------------------------------------------------------------- */

/* For plane p in {0 (gate), 1 (up)} and pair j < n_pairs = t*n_used, with
 * matrix W = mats[p*n_pairs + j] ([n_ff][in_f] in format fmt) and token
 * i = j / n_used:
 *   y[p][j][r]      = scales[p*n_pairs + j] * sum_c W[r][c] * x[i][c]
 *   absmag[p][j][r] = |scales[p*n_pairs + j]| * sum_c |W[r][c] * x[i][c]|
 * y and absmag are [2][n_pairs][n_ff].  Only rows in [row0, row0+nrows) are
 * computed (pass 0, n_ff for all of them); the rest are left untouched. */
int oracle_moe_gate_up(int fmt, const uint8_t *const *mats, const float *scales, const float *x,
                       int64_t in_f, int64_t n_ff, int n_used, int t, int64_t row0, int64_t nrows,
                       double *y, double *absmag, int threads) {
    int64_t rb = oracle_row_bytes(fmt, in_f);
    if (rb == 0 || n_used <= 0 || t <= 0) return -1;
    int64_t n_pairs = (int64_t)t * n_used;
    if (row0 < 0 || nrows < 0 || row0 + nrows > n_ff) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
#endif
    for (int64_t idx = 0; idx < 2 * n_pairs * nrows; ++idx) {
        int64_t mat = idx / nrows;
        int64_t r = row0 + idx % nrows;
        int64_t j = mat % n_pairs;
        int64_t tok = j / n_used;
        double *row = (double *)malloc(sizeof(double) * (size_t)in_f);
        if (!row || oracle_decode_row(fmt, mats[mat] + r * rb, in_f, row) != 0) {
            bad |= 1;
            free(row);
            continue;
        }
        double s = 0.0, a = 0.0;
        for (int64_t c = 0; c < in_f; ++c) {
            double p = row[c] * (double)x[tok * in_f + c];
            s += p;
            a += fabs(p);
        }
        double sc = (double)scales[mat];
        y[mat * n_ff + r] = sc * s;
        if (absmag) absmag[mat * n_ff + r] = fabs(sc) * a;
        free(row);
    }
    (void)threads;
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------- */
/* int8 activations ([memra] main: quantize_q8_1 before the served gate/up   */
/* kernel; the page prints neither, so the block rule is the plain Q8_1     */
/* one: 32 values per block, one scale per block)                           */
/* ---------------------------------------------------------------------- */

/* For every block of 32 consecutive values of a row of x ([rows][k], k a
 * multiple of 32): amax = the largest |x|, d = amax / 127, and every value
 * becomes q = x * (1/d) rounded to the nearest integer, halves away from
 * zero (q = 0 when d = 0).  Every step is one float32 operation, so the
 * integer codes are decided in float32.  d is [rows][k/32], q [rows][k]. */
int oracle_quantize_q8_1(const float *x, int64_t rows, int64_t k, int8_t *q, float *d) {
    if (rows < 0 || k <= 0 || k % 32 != 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const float *xb = x + r * k + 32 * b;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                float a = fabsf(xb[j]);
                if (a > amax) amax = a;
            }
            float db = amax / 127.0f;
            float id = db != 0.0f ? 1.0f / db : 0.0f;
            d[r * (k / 32) + b] = db;
            for (int j = 0; j < 32; ++j) q[r * k + 32 * b + j] = (int8_t)roundf(xb[j] * id);
        }
    }
    return 0;
}

/* The gate/up products of oracle_moe_gate_up with each token's activation
 * given as Q8_1 blocks: x[tok][c] = q[tok][c] * d[tok][c/32], exact in
 * double, the rest unchanged. */
int oracle_moe_gate_up_q8(int fmt, const uint8_t *const *mats, const float *scales, const int8_t *q,
                          const float *d, int64_t in_f, int64_t n_ff, int n_used, int t, int64_t row0,
                          int64_t nrows, double *y, double *absmag, int threads) {
    int64_t rb = oracle_row_bytes(fmt, in_f);
    if (rb == 0 || in_f % 32 != 0 || n_used <= 0 || t <= 0) return -1;
    int64_t n_pairs = (int64_t)t * n_used;
    if (row0 < 0 || nrows < 0 || row0 + nrows > n_ff) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
#endif
    for (int64_t idx = 0; idx < 2 * n_pairs * nrows; ++idx) {
        int64_t mat = idx / nrows;
        int64_t r = row0 + idx % nrows;
        int64_t tok = (mat % n_pairs) / n_used;
        double *row = (double *)malloc(sizeof(double) * (size_t)in_f);
        if (!row || oracle_decode_row(fmt, mats[mat] + r * rb, in_f, row) != 0) {
            bad |= 1;
            free(row);
            continue;
        }
        double s = 0.0, a = 0.0;
        for (int64_t c = 0; c < in_f; ++c) {
            double xv = (double)q[tok * in_f + c] * (double)d[tok * (in_f / 32) + c / 32];
            double p = row[c] * xv;
            s += p;
            a += fabs(p);
        }
        double sc = (double)scales[mat];
        y[mat * n_ff + r] = sc * s;
        if (absmag) absmag[mat * n_ff + r] = fabs(sc) * a;
        free(row);
    }
    (void)threads;
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------- */
/* MoE down projection ([memra] main: the down pass after gate/up)        */
/* ---------------------------------------------------------------------- */

/* For token i < t and output row r < gin, over the token's pairs j = i*n_used
 * + u (u < n_used), with W = mats[j] ([gin][n_ff] in format fmt) and the
 * pair's activation h[j][*] (n_ff values):
 *   y[i][r]      = sum_u scales[j] * sum_c W[r][c] * h[j][c]
 *   absmag[i][r] = sum_u |scales[j]| * sum_c |W[r][c] * h[j][c]|
 * y and absmag are [t][gin].  Only rows in [row0, row0+nrows) are computed
 * (pass 0, gin for all of them); the rest are left untouched. */
int oracle_moe_down(int fmt, const uint8_t *const *mats, const float *scales, const float *h,
                    int64_t n_ff, int64_t gin, int n_used, int t, int64_t row0, int64_t nrows,
                    double *y, double *absmag, int threads) {
    int64_t rb = oracle_row_bytes(fmt, n_ff);
    if (rb == 0 || n_used <= 0 || t <= 0) return -1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > gin) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
#endif
    for (int64_t idx = 0; idx < (int64_t)t * nrows; ++idx) {
        int64_t i = idx / nrows;
        int64_t r = row0 + idx % nrows;
        double *row = (double *)malloc(sizeof(double) * (size_t)n_ff);
        if (!row) {
            bad |= 1;
            continue;
        }
        double s = 0.0, a = 0.0;
        for (int u = 0; u < n_used; ++u) {
            int64_t j = i * n_used + u;
            if (oracle_decode_row(fmt, mats[j] + r * rb, n_ff, row) != 0) {
                bad |= 1;
                break;
            }
            double d = 0.0, m = 0.0;
            for (int64_t c = 0; c < n_ff; ++c) {
                double p = row[c] * (double)h[j * n_ff + c];
                d += p;
                m += fabs(p);
            }
            double sc = (double)scales[j];
            s += sc * d;
            a += fabs(sc) * m;
        }
        y[i * gin + r] = s;
        if (absmag) absmag[i * gin + r] = a;
        free(row);
    }
    (void)threads;
    return bad ? -1 : 0;
}

/* The down projection of oracle_moe_down with each pair's activation given
 * as Q8_1 blocks: h[j][c] = q[j][c] * d[j][c/32], exact in double. */
int oracle_moe_down_q8(int fmt, const uint8_t *const *mats, const float *scales, const int8_t *q,
                       const float *dsc, int64_t n_ff, int64_t gin, int n_used, int t, int64_t row0,
                       int64_t nrows, double *y, double *absmag, int threads) {
    int64_t rb = oracle_row_bytes(fmt, n_ff);
    if (rb == 0 || n_ff % 32 != 0 || n_used <= 0 || t <= 0) return -1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > gin) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
#endif
    for (int64_t idx = 0; idx < (int64_t)t * nrows; ++idx) {
        int64_t i = idx / nrows;
        int64_t r = row0 + idx % nrows;
        double *row = (double *)malloc(sizeof(double) * (size_t)n_ff);
        if (!row) {
            bad |= 1;
            continue;
        }
        double s = 0.0, a = 0.0;
        for (int u = 0; u < n_used; ++u) {
            int64_t j = i * n_used + u;
            if (oracle_decode_row(fmt, mats[j] + r * rb, n_ff, row) != 0) {
                bad |= 1;
                break;
            }
            double dd = 0.0, m = 0.0;
            for (int64_t c = 0; c < n_ff; ++c) {
                double hv = (double)q[j * n_ff + c] * (double)dsc[j * (n_ff / 32) + c / 32];
                double p = row[c] * hv;
                dd += p;
                m += fabs(p);
            }
            double sc = (double)scales[j];
            s += sc * dd;
            a += fabs(sc) * m;
        }
        y[i * gin + r] = s;
        if (absmag) absmag[i * gin + r] = a;
        free(row);
    }
    (void)threads;
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------- */
/* NVFP4 activations for the block-scaled tensor-core product              */
/* ---------------------------------------------------------------------- */

/* The tensor cores' NVFP4 product (tcgen05 kind::mxf4nvf4) takes both
 * operands as E2M1 values with one E4M3 scale per 16; the pages fix no rule
 * for turning an f32 activation into that form (memra quantizes its
 * activations to Q8_1, aprender's prefill names an FP8 activation scratch).
 * Reading, the plainest one that keeps the activation's own NVFP4 groups:
 * per block of 16 consecutive values of a row, scale = the E4M3 value nearest
 * to amax/6 (6 being the largest E2M1 magnitude), code = the E2M1 value
 * nearest to x/scale, both rounding to nearest with ties to the even code and
 * saturating at the format's largest finite value; every step is one float32
 * operation, so the codes are decided in float32.  A block whose scale
 * rounds to zero gets zero codes.  The rows are written as NVFP4 V2 rows. */

/* E4M3FN code (0x00..0x7E) nearest to v >= 0, ties to the even code,
 * saturating at 448 (0x7E). */
uint8_t oracle_e4m3_rn(float v) {
    if (!(v > 0.0f)) return 0;
    uint32_t best = 0;
    double bd = fabs((double)v);
    for (uint32_t c = 1; c <= 0x7Eu; ++c) {
        double d = fabs(oracle_e4m3(c) - (double)v);
        if (d < bd || (d == bd && (c & 1u) == 0)) {
            best = c;
            bd = d;
        }
    }
    return (uint8_t)best;
}

/* E2M1 code (4 bits) nearest to v, ties to the even code, saturating at
 * +-6; the sign bit is v's (a negative value that rounds to zero gives
 * code 8, -0). */
uint8_t oracle_e2m1_rn(float v) {
    uint32_t sign = signbit(v) ? 8u : 0u;
    double a = fabs((double)v);
    uint32_t best = 0;
    double bd = a;
    for (uint32_t c = 1; c <= 7u; ++c) {
        double d = fabs(oracle_e2m1(c) - a);
        if (d < bd || (d == bd && (c & 1u) == 0)) {
            best = c;
            bd = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* x [rows][k] f32 -> rows of NVFP4 V2 ([rows][k/32*18] bytes: k/2 code
 * bytes, element 2j in the low nibble of byte j, then k/16 scale bytes). */
int oracle_quantize_nvfp4_v2(const float *x, int64_t rows, int64_t k, uint8_t *out) {
    if (rows < 0 || k <= 0 || k % 32 != 0) return -1;
    int64_t rb = k / 32 * 18;
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t *row = out + r * rb;
        memset(row, 0, (size_t)rb);
        for (int64_t b = 0; b < k / 16; ++b) {
            const float *xb = x + r * k + 16 * b;
            float amax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(xb[j]);
                if (a > amax) amax = a;
            }
            float t = amax / 6.0f;
            uint8_t sc = oracle_e4m3_rn(t);
            float s = (float)oracle_e4m3(sc);
            row[k / 2 + b] = sc;
            for (int j = 0; j < 16; ++j) {
                uint8_t c = (s == 0.0f) ? 0u : oracle_e2m1_rn(xb[j] / s);
                int64_t e = 16 * b + j;
                row[e / 2] |= (uint8_t)((e % 2 == 0) ? c : (c << 4));
            }
        }
    }
    return 0;
}

/* Threads an OpenMP region would use (1 when built without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Array forms of the scalar decoders, for exhaustive checks over all codes. */
void oracle_fp16_array(const uint16_t *codes, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16(codes[i]);
}
void oracle_e4m3_array(const uint8_t *codes, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3(codes[i]);
}
void oracle_e2m1_array(const uint8_t *codes, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1(codes[i] & 15u);
}
