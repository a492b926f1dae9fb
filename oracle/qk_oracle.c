/*
 * qk_oracle.c -- plain, slow, scalar CPU oracle for GGUF block-quantized
 * weights: unpack, dequantize, fp64 GEMV / GEMM, pack and a plain quantizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * imports this file.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA path: every layout below is restated here from the
 * pages and from the readings listed in the design notes.
 *
 * Sources (page title, section / figure):
 *   [HG]  "Hitchhiker's Guide -- Lab 01: Air-Gapped LLM Serving",
 *         section 11.1 "What quantization actually stores -- block-wise scales"
 *         (w ~ d*q, the Q4_0 block figure: 18 bytes, w ~ d*(q-8); Q8_0 "same
 *         structure with 8-bit codes") and section 11.2 "K-quants decoded"
 *         (the Q4_K super-block figure: 144 bytes, w ~ (d*sc)*q - dmin*m).
 *   [LC]  "12 -- llama.cpp / GGUF / Local Inference Mastery",
 *         "Q4_K_M -- bit layout in exquisite detail" (field order d, dmin,
 *         scales[12], qs[128]; per-sub-block dequantization pseudo-code) and
 *         the "Other k-quants at a glance" table (Q6_K 6.6 bits/weight).
 *   [LK]  "Local LLM inference" (litek8s), "The mmap backend": every block
 *         is dequantized inside the dot product; Q4_K_M mixes Q4_K, Q5_0,
 *         Q6_K and Q8_0.
 *   [EN]  "How LLM Inference Engines Work", "Loading GGUF Models": the Q4_0
 *         dequantizer (low nibbles are elements 0..15, high nibbles 16..31).
 *
 * Field sizes for Q6_K (ql 128 B, qh 64 B, 16 int8 scales, fp16 d) and Q5_0
 * (fp16 d, 4 B high bits, 16 B nibbles) are not on the pages; they come from
 * the workload definition, and the bit placement inside them is a reading
 * (see the per-type comments).  Q5_K appears on the pages only as 5.5-5.7
 * bits/weight on 256-weight super-blocks ([LC] "Other k-quants at a
 * glance"); its whole layout is a reading (the GGUF k-quant one, see
 * unpack_q5_K).  So are Q2_K (2.5-2.6 bits/weight there) and Q3_K (3.4-4.0),
 * see unpack_q2_K and unpack_q3_K.
 *
 * All arithmetic that produces a weight is fp32 in the order the formulas
 * state; dot products accumulate in fp64.  Compile with -ffp-contract=off so
 * that no multiply-add is fused behind the reader's back.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Type ids of the oracle (same numbers as the library's public enum; both
 * sides define them independently). */
enum { OQ_Q4_K = 1, OQ_Q6_K = 2, OQ_Q8_0 = 3, OQ_Q5_0 = 4, OQ_Q4_0 = 5, OQ_Q5_K = 6, OQ_Q2_K = 7, OQ_Q3_K = 8 };

/* ------------------------------------------------------------------------ */
/* Sizes                                                                    */
/* ------------------------------------------------------------------------ */

/* Bytes per block.  Q4_K: 2 (d) + 2 (dmin) + 12 (scales) + 128 (qs) = 144
 * [HG 11.2 figure, LC figure].  Q4_0: 2 + 16 = 18 [HG 11.1 figure].
 * Q8_0: 2 + 32 = 34 [HG 11.1: same structure, 8-bit codes].
 * Q6_K: 128 + 64 + 16 + 2 = 210.  Q5_0: 2 + 4 + 16 = 22. */
int oq_block_bytes(int type) {
    switch (type) {
    case OQ_Q4_K: return 2 + 2 + 12 + 128;
    case OQ_Q6_K: return 128 + 64 + 16 + 2;
    case OQ_Q8_0: return 2 + 32;
    case OQ_Q5_0: return 2 + 4 + 16;
    case OQ_Q4_0: return 2 + 16;
    case OQ_Q5_K: return 2 + 2 + 12 + 32 + 128;
    case OQ_Q2_K: return 16 + 64 + 2 + 2;
    case OQ_Q3_K: return 32 + 64 + 12 + 2;
    default: return -1;
    }
}

/* Weights per block: 256 for the K-quant super-blocks [HG 11.2], 32 for the
 * classic blocks [HG 11.1]. */
int oq_block_elems(int type) {
    switch (type) {
    case OQ_Q4_K: case OQ_Q6_K: case OQ_Q5_K: case OQ_Q2_K: case OQ_Q3_K: return 256;
    case OQ_Q8_0: case OQ_Q5_0: case OQ_Q4_0: return 32;
    default: return -1;
    }
}

/* ------------------------------------------------------------------------ */
/* Floating-point formats, written from their definitions                   */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 = zero / subnormal (f * 2^-24), 31 = Inf / NaN. */
float oq_half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return (float)(sign ? -v : v);
}

/* Round a finite value to binary16, ties to even; overflow gives Inf. */
uint16_t oq_float_to_half(float xf) {
    double x = (double)xf;
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000 : 0);
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7E00);
    if (isinf(x)) return (uint16_t)(sign | 0x7C00);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);              /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;             /* 2^e <= a < 2^(e+1) */
    if (e < -14) e = -14;       /* subnormal range shares the quantum 2^-24 */
    double quantum = ldexp(1.0, e - 10);
    double q = rint(a / quantum) * quantum;   /* default mode: ties to even */
    if (q >= 65520.0) return (uint16_t)(sign | 0x7C00);
    if (q < ldexp(1.0, -14)) {
        return (uint16_t)(sign | (uint16_t)(q / ldexp(1.0, -24)));
    }
    frexp(q, &e2);
    e = e2 - 1;
    uint16_t frac = (uint16_t)(q / ldexp(1.0, e - 10) - 1024.0);
    return (uint16_t)(sign | ((e + 15) << 10) | frac);
}

/* bfloat16 is the top half of a binary32: 8 exponent bits, 7 fraction bits.
 * Rounding keeps 8 significant bits, ties to even; the subnormal quantum is
 * 2^-133.  NaN stays NaN. */
uint16_t oq_float_to_bf16(float xf) {
    if (isnan(xf)) return 0x7FC0;
    double x = (double)xf;
    double a = fabs(x);
    uint32_t sbit = signbit(x) ? 0x80000000u : 0u;
    float r;
    if (a == 0.0 || isinf(x)) {
        r = (float)a;
    } else {
        int e2;
        frexp(a, &e2);
        int e = e2 - 1;
        if (e < -126) e = -126;
        double quantum = ldexp(1.0, e - 7);
        double q = rint(a / quantum) * quantum;
        r = (float)q;           /* exact, or Inf past the largest finite */
    }
    uint32_t bits;
    memcpy(&bits, &r, 4);
    bits |= sbit;
    return (uint16_t)(bits >> 16);
}

float oq_bf16_to_float(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 255); p[1] = (uint8_t)(v >> 8); }

/* ------------------------------------------------------------------------ */
/* Unpack: bytes -> integer codes, sub-block scales / mins, fp32 d / dmin    */
/* ------------------------------------------------------------------------ */

/* Q4_K super-block [HG 11.2 figure; LC figure and pseudo-code].
 * Bytes 0-1 d, 2-3 dmin (binary16, little-endian), 4-15 the 8 packed
 * (6-bit scale, 6-bit min) pairs, 16-143 the 256 4-bit codes.
 * The pages say only that the twelve bytes hold 8 x (6-bit scale + 6-bit
 * min); the reading adopted is the k-quant packing the pages cite:
 *   sub-blocks 0..3:  sc = s[j] & 63,   m = s[j+4] & 63
 *   sub-blocks 4..7:  sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
 *                     m  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
 * Code order: weight n lives in byte qs[32*(n/64) + n%32], low nibble when
 * (n/32) is even, high nibble when odd -- the same low-half / high-half
 * nibble convention as the Q4_0 dequantizer in [EN], applied per 32 bytes.
 * Weight n belongs to sub-block n/32. */
static void unpack_q4_K(const uint8_t* b, int16_t* q, int16_t* sc, uint8_t* mn, float* d, float* dmin) {
    const uint8_t* s = b + 4;
    const uint8_t* qs = b + 16;
    *d = oq_half_to_float(rd16(b));
    *dmin = oq_half_to_float(rd16(b + 2));
    for (int j = 0; j < 8; j++) {
        if (j < 4) {
            sc[j] = (int16_t)(s[j] & 63);
            mn[j] = (uint8_t)(s[j + 4] & 63);
        } else {
            sc[j] = (int16_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));
            mn[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
        }
    }
    for (int n = 0; n < 256; n++) {
        int c = n / 64, h = (n / 32) % 2, l = n % 32;
        q[n] = (int16_t)((qs[32 * c + l] >> (4 * h)) & 15);
    }
}

/* Q5_K super-block (176 bytes = 5.5 bits/weight, the low end of [LC]'s
 * 5.5-5.7): a Q4_K super-block with a fifth code bit per weight.  Reading
 * (the GGUF k-quant layout): bytes 0-1 d, 2-3 dmin, 4-15 the eight
 * (6-bit scale, 6-bit min) pairs packed exactly as in Q4_K, 16-47 qh (one
 * high bit per weight), 48-175 qs (the low 4 bits, placed as Q4_K's codes).
 * Weight n, with c = n/64, h = (n/32)%2, l = n%32:
 *   lo4 = (qs[32c + l] >> 4h) & 15,   hb = (qh[l] >> (2c + h)) & 1,
 *   q = lo4 | hb << 4   (0..31),       w = (d*sc)*q - dmin*m of sub-block n/32. */
static void unpack_q5_K(const uint8_t* b, int16_t* q, int16_t* sc, uint8_t* mn, float* d, float* dmin) {
    const uint8_t* s = b + 4;
    const uint8_t* qh = b + 16;
    const uint8_t* qs = b + 48;
    *d = oq_half_to_float(rd16(b));
    *dmin = oq_half_to_float(rd16(b + 2));
    for (int j = 0; j < 8; j++) {
        if (j < 4) {
            sc[j] = (int16_t)(s[j] & 63);
            mn[j] = (uint8_t)(s[j + 4] & 63);
        } else {
            sc[j] = (int16_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));
            mn[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
        }
    }
    for (int n = 0; n < 256; n++) {
        int c = n / 64, h = (n / 32) % 2, l = n % 32;
        int lo4 = (qs[32 * c + l] >> (4 * h)) & 15;
        int hb = (qh[l] >> (2 * c + h)) & 1;
        q[n] = (int16_t)(lo4 | (hb << 4));
    }
}

/* Q2_K super-block (84 bytes = 2.625 bits/weight, [LC]'s "2.5-2.6"):
 * sixteen 16-weight groups, each with a 4-bit scale and a 4-bit min.
 * Reading (the GGUF k-quant layout): bytes 0-15 one byte per group (scale in
 * the low nibble, min in the high nibble), 16-79 qs (2-bit codes), 80-81 d,
 * 82-83 dmin.  Weight n, with t = n/128, j = (n%128)/32, l = n%32:
 *   q = (qs[32t + l] >> 2j) & 3   (0..3),   group g = n/16,
 *   w = (d*sc_g)*q - dmin*m_g. */
static void unpack_q2_K(const uint8_t* b, int16_t* q, int16_t* sc, uint8_t* mn, float* d, float* dmin) {
    const uint8_t* qs = b + 16;
    *d = oq_half_to_float(rd16(b + 80));
    *dmin = oq_half_to_float(rd16(b + 82));
    for (int g = 0; g < 16; g++) {
        sc[g] = (int16_t)(b[g] & 15);
        mn[g] = (uint8_t)(b[g] >> 4);
    }
    for (int n = 0; n < 256; n++) {
        int t = n / 128, j = (n % 128) / 32, l = n % 32;
        q[n] = (int16_t)((qs[32 * t + l] >> (2 * j)) & 3);
    }
}

/* Q3_K super-block (110 bytes = 3.4375 bits/weight, within [LC]'s
 * "3.4-4.0"): sixteen 16-weight groups with signed 6-bit scales, 3-bit
 * codes.  Reading (the GGUF k-quant layout): bytes 0-31 hmask, 32-95 qs
 * (low 2 bits of each code), 96-107 the sixteen 6-bit scales, 108-109 d.
 * Weight n, with t = n/128, j = (n%128)/32, l = n%32:
 *   lo2 = (qs[32t + l] >> 2j) & 3,  hb = (hmask[l] >> (4t + j)) & 1,
 *   q = lo2 - 4 when hb is clear, lo2 when set   (-4..3).
 * Scale of group g (0..15), from s = bytes 96..107: the low 4 bits are the
 * low (g < 8) or high (g >= 8) nibble of s[g % 8], the high 2 bits are bits
 * 2(g/4), 2(g/4)+1 of s[8 + g % 4]; the 6-bit value minus 32 is the scale
 * (-32..31).  w = (d*sc_g)*q. */
static void unpack_q3_K(const uint8_t* b, int16_t* q, int16_t* sc, float* d) {
    const uint8_t* hm = b;
    const uint8_t* qs = b + 32;
    const uint8_t* s = b + 96;
    *d = oq_half_to_float(rd16(b + 108));
    for (int g = 0; g < 16; g++) {
        int lo4 = (s[g % 8] >> (4 * (g / 8))) & 15;
        int hi2 = (s[8 + g % 4] >> (2 * (g / 4))) & 3;
        sc[g] = (int16_t)((lo4 | (hi2 << 4)) - 32);
    }
    for (int n = 0; n < 256; n++) {
        int t = n / 128, j = (n % 128) / 32, l = n % 32;
        int lo2 = (qs[32 * t + l] >> (2 * j)) & 3;
        int hb = (hm[l] >> (4 * t + j)) & 1;
        q[n] = (int16_t)(hb ? lo2 : lo2 - 4);
    }
}

/* Q6_K super-block (210 bytes): bytes 0-127 ql (low 4 bits of each code),
 * 128-191 qh (high 2 bits), 192-207 sixteen int8 sub-block scales (one per
 * 16 weights), 208-209 d.  Reading of the bit placement: within half
 * t = n/128, with r = n%128, l = r%32, g = r/32,
 *   lo4 = ql[64t + l + 32*(g&1)], low nibble for g in {0,1}, high for {2,3}
 *   hi2 = (qh[32t + l] >> 2g) & 3,     q = lo4 | hi2 << 4   (0..63)
 * and the weight is d * sc[n/16] * (q - 32) (symmetric offset, by analogy
 * with Q4_0's q - 8 in [HG 11.1]). */
static void unpack_q6_K(const uint8_t* b, int16_t* q, int16_t* sc, float* d) {
    const uint8_t* ql = b;
    const uint8_t* qh = b + 128;
    const int8_t* scales = (const int8_t*)(b + 192);
    *d = oq_half_to_float(rd16(b + 208));
    for (int j = 0; j < 16; j++) sc[j] = scales[j];
    for (int n = 0; n < 256; n++) {
        int t = n / 128, r = n % 128, l = r % 32, g = r / 32;
        int byte = ql[64 * t + l + 32 * (g & 1)];
        int lo4 = (g < 2) ? (byte & 15) : (byte >> 4);
        int hi2 = (qh[32 * t + l] >> (2 * g)) & 3;
        q[n] = (int16_t)(lo4 | (hi2 << 4));
    }
}

/* Q8_0 (34 bytes): bytes 0-1 d, 2-33 thirty-two signed 8-bit codes;
 * w = d * q [HG 11.1]. */
static void unpack_q8_0(const uint8_t* b, int16_t* q, float* d) {
    *d = oq_half_to_float(rd16(b));
    for (int j = 0; j < 32; j++) q[j] = (int16_t)(int8_t)b[2 + j];
}

/* Q5_0 (22 bytes): bytes 0-1 d, 2-5 a little-endian 32-bit word of fifth
 * bits, 6-21 sixteen bytes of nibbles.  Element j < 16 takes the low nibble
 * of qs[j], element j + 16 the high nibble (the [EN] Q4_0 convention); bit j
 * of the word is element j's fifth bit.  w = d * (q - 16). */
static void unpack_q5_0(const uint8_t* b, int16_t* q, float* d) {
    *d = oq_half_to_float(rd16(b));
    uint32_t qh = (uint32_t)b[2] | ((uint32_t)b[3] << 8) | ((uint32_t)b[4] << 16) | ((uint32_t)b[5] << 24);
    const uint8_t* qs = b + 6;
    for (int j = 0; j < 16; j++) {
        q[j] = (int16_t)((qs[j] & 15) | (((qh >> j) & 1) << 4));
        q[j + 16] = (int16_t)((qs[j] >> 4) | (((qh >> (j + 16)) & 1) << 4));
    }
}

/* Q4_0 (18 bytes) [HG 11.1 figure; EN "Loading GGUF Models"]: bytes 0-1 d,
 * then 16 bytes; element j < 16 is the low nibble of byte j, element j + 16
 * the high nibble.  w = d * (q - 8). */
static void unpack_q4_0(const uint8_t* b, int16_t* q, float* d) {
    *d = oq_half_to_float(rd16(b));
    for (int j = 0; j < 16; j++) {
        q[j] = (int16_t)(b[2 + j] & 15);
        q[j + 16] = (int16_t)(b[2 + j] >> 4);
    }
}

/* Unpack nblocks blocks.  codes: [nblocks * block_elems]; sc: [nblocks * 16]
 * (Q4_K / Q5_K use 8 slots, Q6_K / Q2_K / Q3_K 16; unused slots are 0);
 * mins: [nblocks * 16] (Q4_K / Q5_K 8 slots, Q2_K 16; 0 elsewhere); d, dmin:
 * [nblocks].  Any output pointer may be NULL. */
int oq_unpack(int type, const uint8_t* blocks, int64_t nblocks,
              int16_t* codes, int16_t* sc, uint8_t* mins, float* d, float* dmin) {
    int bb = oq_block_bytes(type), be = oq_block_elems(type);
    if (bb < 0) return -1;
    for (int64_t i = 0; i < nblocks; i++) {
        const uint8_t* b = blocks + i * bb;
        int16_t q[256], s[16];
        uint8_t m[16];
        float dd = 0.0f, dm = 0.0f;
        memset(s, 0, sizeof s);
        memset(m, 0, sizeof m);
        switch (type) {
        case OQ_Q4_K: unpack_q4_K(b, q, s, m, &dd, &dm); break;
        case OQ_Q6_K: unpack_q6_K(b, q, s, &dd); break;
        case OQ_Q8_0: unpack_q8_0(b, q, &dd); break;
        case OQ_Q5_0: unpack_q5_0(b, q, &dd); break;
        case OQ_Q4_0: unpack_q4_0(b, q, &dd); break;
        case OQ_Q5_K: unpack_q5_K(b, q, s, m, &dd, &dm); break;
        case OQ_Q2_K: unpack_q2_K(b, q, s, m, &dd, &dm); break;
        case OQ_Q3_K: unpack_q3_K(b, q, s, &dd); break;
        }
        if (codes) memcpy(codes + i * be, q, (size_t)be * sizeof(int16_t));
        if (sc) memcpy(sc + i * 16, s, sizeof s);
        if (mins) memcpy(mins + i * 16, m, sizeof m);
        if (d) d[i] = dd;
        if (dmin) dmin[i] = dm;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantize (fp32, per the formulas, in the order they are written)       */
/* ------------------------------------------------------------------------ */

/* One block -> block_elems fp32 weights.
 *   Q4_K: ds = d*sc, dm = dmin*m, w = ds*q - dm   [HG 11.2, LC pseudo-code]
 *   Q5_K: the same with 5-bit codes
 *   Q2_K: the same per 16-weight group with 2-bit codes and 4-bit sc, m
 *   Q3_K: w = (d*sc) * q, signed sc and q
 *   Q6_K: w = (d*sc) * (q - 32)
 *   Q8_0: w = d * q                                [HG 11.1]
 *   Q5_0: w = d * (q - 16)
 *   Q4_0: w = d * (q - 8)                          [HG 11.1, EN]          */
static void dequant_block(int type, const uint8_t* b, float* w) {
    int16_t q[256], s[16];
    uint8_t m[16];
    float d = 0.0f, dmin = 0.0f;
    switch (type) {
    case OQ_Q4_K:
        unpack_q4_K(b, q, s, m, &d, &dmin);
        for (int n = 0; n < 256; n++) {
            float ds = d * (float)s[n / 32];
            float dm = dmin * (float)m[n / 32];
            float t = ds * (float)q[n];
            w[n] = t - dm;
        }
        break;
    case OQ_Q5_K:
        unpack_q5_K(b, q, s, m, &d, &dmin);
        for (int n = 0; n < 256; n++) {
            float ds = d * (float)s[n / 32];
            float dm = dmin * (float)m[n / 32];
            float t = ds * (float)q[n];
            w[n] = t - dm;
        }
        break;
    case OQ_Q2_K:
        unpack_q2_K(b, q, s, m, &d, &dmin);
        for (int n = 0; n < 256; n++) {
            float ds = d * (float)s[n / 16];
            float dm = dmin * (float)m[n / 16];
            float t = ds * (float)q[n];
            w[n] = t - dm;
        }
        break;
    case OQ_Q3_K:
        unpack_q3_K(b, q, s, &d);
        for (int n = 0; n < 256; n++) {
            float ds = d * (float)s[n / 16];
            w[n] = ds * (float)q[n];
        }
        break;
    case OQ_Q6_K:
        unpack_q6_K(b, q, s, &d);
        for (int n = 0; n < 256; n++) {
            float ds = d * (float)s[n / 16];
            w[n] = ds * (float)(q[n] - 32);
        }
        break;
    case OQ_Q8_0:
        unpack_q8_0(b, q, &d);
        for (int n = 0; n < 32; n++) w[n] = d * (float)q[n];
        break;
    case OQ_Q5_0:
        unpack_q5_0(b, q, &d);
        for (int n = 0; n < 32; n++) w[n] = d * (float)(q[n] - 16);
        break;
    case OQ_Q4_0:
        unpack_q4_0(b, q, &d);
        for (int n = 0; n < 32; n++) w[n] = d * (float)(q[n] - 8);
        break;
    }
}

static int check_shape(int type, int64_t rows, int64_t cols) {
    int be = oq_block_elems(type);
    if (be < 0) return -1;
    if (rows < 0 || cols < 0 || cols % be != 0) return -2;
    return 0;
}

/* W is [rows, cols] row-major in blocks along cols: row r starts at byte
 * r * (cols / block_elems) * block_bytes.  out: fp32 [rows, cols]. */
int oq_dequant(int type, const uint8_t* W, int64_t rows, int64_t cols, float* out) {
    int rc = check_shape(type, rows, cols);
    if (rc) return rc;
    int bb = oq_block_bytes(type), be = oq_block_elems(type);
    int64_t nb = cols / be;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t i = 0; i < nb; i++)
            dequant_block(type, W + (r * nb + i) * bb, out + r * cols + i * be);
    return 0;
}

static void dequant_row(int type, const uint8_t* W, int64_t cols, int64_t r, float* row) {
    int bb = oq_block_bytes(type), be = oq_block_elems(type);
    int64_t nb = cols / be;
    for (int64_t i = 0; i < nb; i++)
        dequant_block(type, W + (r * nb + i) * bb, row + i * be);
}

/* ------------------------------------------------------------------------ */
/* Matrix products in fp64 over the exactly dequantized weights             */
/* ------------------------------------------------------------------------ */

/* y[m, n] = sum_k w[n, k] * x[m, k] in fp64, S[m, n] = sum_k |w[n,k]*x[m,k]|
 * (the scale of the tolerance).  x fp32 [M, cols]; y, S fp64 [M, rows].
 * The weights are dequantized inside the dot product, row by row [LK]. */
int oq_gemv(int type, const uint8_t* W, int64_t rows, int64_t cols,
            const float* x, int64_t M, double* y, double* S) {
    int rc = check_shape(type, rows, cols);
    if (rc) return rc;
    float* row = (float*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(float));
    if (!row) return -3;
    for (int64_t n = 0; n < rows; n++) {
        dequant_row(type, W, cols, n, row);
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, s = 0.0;
            const float* xm = x + m * cols;
            for (int64_t k = 0; k < cols; k++) {
                double p = (double)row[k] * (double)xm[k];
                acc += p;
                s += fabs(p);
            }
            y[m * rows + n] = acc;
            if (S) S[m * rows + n] = s;
        }
    }
    free(row);
    return 0;
}

/* Same as oq_gemv for a bf16 activation matrix X [M, cols] given as raw
 * bfloat16 bits: the reference for the tensor-core GEMM, whose activations
 * are bf16 and whose weights are exact. */
int oq_gemm_bf16(int type, const uint8_t* W, int64_t rows, int64_t cols,
                 const uint16_t* X, int64_t M, double* Y, double* S) {
    int rc = check_shape(type, rows, cols);
    if (rc) return rc;
    float* row = (float*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(float));
    if (!row) return -3;
    for (int64_t n = 0; n < rows; n++) {
        dequant_row(type, W, cols, n, row);
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, s = 0.0;
            const uint16_t* xm = X + m * cols;
            for (int64_t k = 0; k < cols; k++) {
                double p = (double)row[k] * (double)oq_bf16_to_float(xm[k]);
                acc += p;
                s += fabs(p);
            }
            Y[m * rows + n] = acc;
            if (S) S[m * rows + n] = s;
        }
    }
    free(row);
    return 0;
}

/* Selected outputs only: for e in 0..count-1, the (mi[e], ni[e]) entry of
 * the GEMV (X fp32) or, when xb is non-NULL, of the bf16 GEMM. */
int oq_entries(int type, const uint8_t* W, int64_t rows, int64_t cols,
               const float* x, const uint16_t* xb, int64_t M,
               const int64_t* mi, const int64_t* ni, int64_t count,
               double* y, double* S) {
    int rc = check_shape(type, rows, cols);
    if (rc) return rc;
    float* row = (float*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(float));
    if (!row) return -3;
    int64_t cached = -1;
    for (int64_t e = 0; e < count; e++) {
        int64_t m = mi[e], n = ni[e];
        if (m < 0 || m >= M || n < 0 || n >= rows) { free(row); return -4; }
        if (n != cached) { dequant_row(type, W, cols, n, row); cached = n; }
        double acc = 0.0, s = 0.0;
        for (int64_t k = 0; k < cols; k++) {
            double xv = xb ? (double)oq_bf16_to_float(xb[m * cols + k]) : (double)x[m * cols + k];
            double p = (double)row[k] * xv;
            acc += p;
            s += fabs(p);
        }
        y[e] = acc;
        if (S) S[e] = s;
    }
    free(row);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Pack: the exact inverse of unpack (codes, scales, mins, fp16 bits)       */
/* ------------------------------------------------------------------------ */

/* codes [nblocks * block_elems]: Q4_K 0..15, Q5_K 0..31, Q6_K 0..63, Q8_0
 * -128..127, Q5_0 0..31, Q4_0 0..15, Q2_K 0..3, Q3_K -4..3.  sc [nblocks*16]:
 * Q4_K / Q5_K 0..63 (8 used), Q6_K -128..127, Q2_K 0..15, Q3_K -32..31.
 * mins [nblocks*16]: Q4_K / Q5_K 0..63 (8 used), Q2_K 0..15.
 * d_bits / dmin_bits: binary16.
 * Returns -5 when a field is out of range. */
int oq_pack(int type, int64_t nblocks, const int16_t* codes, const int16_t* sc,
            const uint8_t* mins, const uint16_t* d_bits, const uint16_t* dmin_bits,
            uint8_t* out) {
    int bb = oq_block_bytes(type), be = oq_block_elems(type);
    if (bb < 0) return -1;
    for (int64_t i = 0; i < nblocks; i++) {
        uint8_t* b = out + i * bb;
        const int16_t* q = codes + i * be;
        memset(b, 0, (size_t)bb);
        switch (type) {
        case OQ_Q4_K:
        case OQ_Q5_K: {
            const int five = type == OQ_Q5_K;
            const int16_t* s = sc + i * 16;
            const uint8_t* m = mins + i * 16;
            uint8_t* S = b + 4;
            uint8_t* qh = b + 16;                  /* Q5_K only */
            uint8_t* qs = b + (five ? 48 : 16);
            wr16(b, d_bits[i]);
            wr16(b + 2, dmin_bits[i]);
            for (int j = 0; j < 8; j++)
                if (s[j] < 0 || s[j] > 63 || m[j] > 63) return -5;
            for (int j = 0; j < 4; j++) {
                S[j] = (uint8_t)((s[j] & 63) | ((s[j + 4] >> 4) << 6));
                S[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
                S[j + 8] = (uint8_t)((s[j + 4] & 15) | ((m[j + 4] & 15) << 4));
            }
            for (int n = 0; n < 256; n++) {
                if (q[n] < 0 || q[n] > (five ? 31 : 15)) return -5;
                int c = n / 64, h = (n / 32) % 2, l = n % 32;
                qs[32 * c + l] |= (uint8_t)((q[n] & 15) << (4 * h));
                if (five) qh[l] |= (uint8_t)((q[n] >> 4) << (2 * c + h));
            }
            break;
        }
        case OQ_Q2_K: {
            const int16_t* s = sc + i * 16;
            const uint8_t* m = mins + i * 16;
            for (int g = 0; g < 16; g++) {
                if (s[g] < 0 || s[g] > 15 || m[g] > 15) return -5;
                b[g] = (uint8_t)(s[g] | (m[g] << 4));
            }
            for (int n = 0; n < 256; n++) {
                if (q[n] < 0 || q[n] > 3) return -5;
                int t = n / 128, j = (n % 128) / 32, l = n % 32;
                b[16 + 32 * t + l] |= (uint8_t)(q[n] << (2 * j));
            }
            wr16(b + 80, d_bits[i]);
            wr16(b + 82, dmin_bits[i]);
            break;
        }
        case OQ_Q3_K: {
            const int16_t* s = sc + i * 16;
            for (int g = 0; g < 16; g++) {
                if (s[g] < -32 || s[g] > 31) return -5;
                int v = s[g] + 32;
                b[96 + g % 8] |= (uint8_t)((v & 15) << (4 * (g / 8)));
                b[104 + g % 4] |= (uint8_t)((v >> 4) << (2 * (g / 4)));
            }
            for (int n = 0; n < 256; n++) {
                if (q[n] < -4 || q[n] > 3) return -5;
                int t = n / 128, j = (n % 128) / 32, l = n % 32;
                int hb = q[n] >= 0, lo2 = hb ? q[n] : q[n] + 4;
                b[32 + 32 * t + l] |= (uint8_t)(lo2 << (2 * j));
                b[l] |= (uint8_t)(hb << (4 * t + j));
            }
            wr16(b + 108, d_bits[i]);
            break;
        }
        case OQ_Q6_K: {
            const int16_t* s = sc + i * 16;
            uint8_t* ql = b;
            uint8_t* qh = b + 128;
            for (int j = 0; j < 16; j++) {
                if (s[j] < -128 || s[j] > 127) return -5;
                b[192 + j] = (uint8_t)(int8_t)s[j];
            }
            wr16(b + 208, d_bits[i]);
            for (int n = 0; n < 256; n++) {
                if (q[n] < 0 || q[n] > 63) return -5;
                int t = n / 128, r = n % 128, l = r % 32, g = r / 32;
                int lo4 = q[n] & 15, hi2 = q[n] >> 4;
                ql[64 * t + l + 32 * (g & 1)] |= (uint8_t)(g < 2 ? lo4 : lo4 << 4);
                qh[32 * t + l] |= (uint8_t)(hi2 << (2 * g));
            }
            break;
        }
        case OQ_Q8_0:
            wr16(b, d_bits[i]);
            for (int j = 0; j < 32; j++) {
                if (q[j] < -128 || q[j] > 127) return -5;
                b[2 + j] = (uint8_t)(int8_t)q[j];
            }
            break;
        case OQ_Q5_0: {
            uint32_t qh = 0;
            wr16(b, d_bits[i]);
            for (int j = 0; j < 32; j++)
                if (q[j] < 0 || q[j] > 31) return -5;
            for (int j = 0; j < 16; j++) {
                b[6 + j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
                qh |= (uint32_t)(q[j] >> 4) << j;
                qh |= (uint32_t)(q[j + 16] >> 4) << (j + 16);
            }
            b[2] = (uint8_t)(qh & 255);
            b[3] = (uint8_t)((qh >> 8) & 255);
            b[4] = (uint8_t)((qh >> 16) & 255);
            b[5] = (uint8_t)(qh >> 24);
            break;
        }
        case OQ_Q4_0:
            wr16(b, d_bits[i]);
            for (int j = 0; j < 32; j++)
                if (q[j] < 0 || q[j] > 15) return -5;
            for (int j = 0; j < 16; j++)
                b[2 + j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
            break;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* A plain quantizer (input generation only; off the hot path)              */
/* ------------------------------------------------------------------------ */

/* clamp(round(v), lo, hi): round half away from zero in fp32, clamp while
 * still a float (so no out-of-range float reaches the int conversion; a NaN
 * quotient takes the low end), then convert. */
static int qclamp(float v, int lo, int hi) {
    float r = roundf(v);
    if (!(r >= (float)lo)) r = (float)lo;
    if (r > (float)hi) r = (float)hi;
    return (int)r;
}

/* Deterministic min/max quantizer.  The pages name the k-quant quantizer
 * (llama.cpp's quantize_row_q4_K) but do not give it; this is the plainest
 * scheme that fills every field:
 *   Q4_K per 32-weight sub-block: mn = min(0, min w), sc_f = (max w - mn)/15,
 *        m_f = -mn; d = max sc_f / 63, dmin = max m_f / 63 (stored fp16);
 *        sc = round(sc_f/d), m = round(m_f/dmin) in 0..63;
 *        q = round((w + dmin*m) / (d*sc)) in 0..15.
 *   Q5_K: the same with 31 in place of 15 (codes 0..31).
 *   Q2_K per 16-weight group: the Q4_K scheme with 3 steps and 4-bit scale
 *        and min (d = max sc_f / 15, dmin = max m_f / 15, codes 0..3).
 *   Q3_K per 16 weights: s = max|w|/4; d = max s / 31; sc = round(s/d) in
 *        -32..31; q = round(w / (d*sc)) in -4..3.
 *   Q6_K per 16 weights: s = max|w|/32; d = max s / 127; sc = round(s/d);
 *        q = round(w / (d*sc)) + 32 in 0..63.
 *   Q8_0: d = max|w|/127, q = round(w/d) in -128..127.
 *   Q5_0: d = max|w|/15,  q = round(w/d) + 16 in 0..31.
 *   Q4_0: d = max|w|/7,   q = round(w/d) + 8 in 0..15.
 * All in fp32, each quotient an IEEE division; round() is half away from
 * zero and the clamp is applied before the conversion to an integer (a NaN
 * quotient gives the lowest code).  A zero divisor gives the zero code. */
int oq_quantize(int type, const float* w, int64_t rows, int64_t cols, uint8_t* out) {
    int rc = check_shape(type, rows, cols);
    if (rc) return rc;
    int bb = oq_block_bytes(type), be = oq_block_elems(type);
    int64_t nblk = rows * (cols / be);
    for (int64_t i = 0; i < nblk; i++) {
        const float* x = w + i * be;
        int16_t q[256], s[16];
        uint8_t m[16];
        uint16_t db = 0, dmb = 0;
        memset(s, 0, sizeof s);
        memset(m, 0, sizeof m);
        if (type == OQ_Q4_K || type == OQ_Q5_K) {
            const int top = type == OQ_Q5_K ? 31 : 15;
            float scf[8], mf[8], maxsc = 0.0f, maxm = 0.0f;
            for (int j = 0; j < 8; j++) {
                float lo = 0.0f, hi = x[32 * j];
                for (int l = 0; l < 32; l++) {
                    float v = x[32 * j + l];
                    if (v < lo) lo = v;
                    if (v > hi) hi = v;
                }
                scf[j] = (hi - lo) / (float)top;
                mf[j] = -lo;
                if (scf[j] > maxsc) maxsc = scf[j];
                if (mf[j] > maxm) maxm = mf[j];
            }
            db = oq_float_to_half(maxsc / 63.0f);
            dmb = oq_float_to_half(maxm / 63.0f);
            float d = oq_half_to_float(db), dmin = oq_half_to_float(dmb);
            for (int j = 0; j < 8; j++) {
                s[j] = (int16_t)(d > 0.0f ? qclamp(scf[j] / d, 0, 63) : 0);
                m[j] = (uint8_t)(dmin > 0.0f ? qclamp(mf[j] / dmin, 0, 63) : 0);
                float ds = d * (float)s[j];
                float dm = dmin * (float)m[j];
                for (int l = 0; l < 32; l++) {
                    float v = x[32 * j + l];
                    q[32 * j + l] = (int16_t)(ds > 0.0f ? qclamp((v + dm) / ds, 0, top) : 0);
                }
            }
        } else if (type == OQ_Q2_K) {
            float scf[16], mf[16], maxsc = 0.0f, maxm = 0.0f;
            for (int g = 0; g < 16; g++) {
                float lo = 0.0f, hi = x[16 * g];
                for (int l = 0; l < 16; l++) {
                    float v = x[16 * g + l];
                    if (v < lo) lo = v;
                    if (v > hi) hi = v;
                }
                scf[g] = (hi - lo) / 3.0f;
                mf[g] = -lo;
                if (scf[g] > maxsc) maxsc = scf[g];
                if (mf[g] > maxm) maxm = mf[g];
            }
            db = oq_float_to_half(maxsc / 15.0f);
            dmb = oq_float_to_half(maxm / 15.0f);
            float d = oq_half_to_float(db), dmin = oq_half_to_float(dmb);
            for (int g = 0; g < 16; g++) {
                s[g] = (int16_t)(d > 0.0f ? qclamp(scf[g] / d, 0, 15) : 0);
                m[g] = (uint8_t)(dmin > 0.0f ? qclamp(mf[g] / dmin, 0, 15) : 0);
                float ds = d * (float)s[g];
                float dm = dmin * (float)m[g];
                for (int l = 0; l < 16; l++) {
                    float v = x[16 * g + l];
                    q[16 * g + l] = (int16_t)(ds > 0.0f ? qclamp((v + dm) / ds, 0, 3) : 0);
                }
            }
        } else if (type == OQ_Q3_K) {
            float sf[16], maxs = 0.0f;
            for (int g = 0; g < 16; g++) {
                float a = 0.0f;
                for (int l = 0; l < 16; l++) {
                    float v = fabsf(x[16 * g + l]);
                    if (v > a) a = v;
                }
                sf[g] = a / 4.0f;
                if (sf[g] > maxs) maxs = sf[g];
            }
            db = oq_float_to_half(maxs / 31.0f);
            float d = oq_half_to_float(db);
            for (int g = 0; g < 16; g++) {
                s[g] = (int16_t)(d > 0.0f ? qclamp(sf[g] / d, -32, 31) : 0);
                float ds = d * (float)s[g];
                for (int l = 0; l < 16; l++) {
                    float v = x[16 * g + l];
                    q[16 * g + l] = (int16_t)(ds != 0.0f ? qclamp(v / ds, -4, 3) : 0);
                }
            }
        } else if (type == OQ_Q6_K) {
            float sf[16], maxs = 0.0f;
            for (int j = 0; j < 16; j++) {
                float a = 0.0f;
                for (int l = 0; l < 16; l++) {
                    float v = fabsf(x[16 * j + l]);
                    if (v > a) a = v;
                }
                sf[j] = a / 32.0f;
                if (sf[j] > maxs) maxs = sf[j];
            }
            db = oq_float_to_half(maxs / 127.0f);
            float d = oq_half_to_float(db);
            for (int j = 0; j < 16; j++) {
                s[j] = (int16_t)(d > 0.0f ? qclamp(sf[j] / d, -128, 127) : 0);
                float ds = d * (float)s[j];
                for (int l = 0; l < 16; l++) {
                    float v = x[16 * j + l];
                    q[16 * j + l] = (int16_t)(ds != 0.0f ? qclamp(v / ds, -32, 31) + 32 : 32);
                }
            }
        } else {
            float a = 0.0f;
            for (int l = 0; l < 32; l++) {
                float v = fabsf(x[l]);
                if (v > a) a = v;
            }
            float div = (type == OQ_Q8_0) ? 127.0f : (type == OQ_Q5_0 ? 15.0f : 7.0f);
            int off = (type == OQ_Q8_0) ? 0 : (type == OQ_Q5_0 ? 16 : 8);
            int lo = (type == OQ_Q8_0) ? -128 : 0;
            int hi = (type == OQ_Q8_0) ? 127 : (type == OQ_Q5_0 ? 31 : 15);
            db = oq_float_to_half(a / div);
            float d = oq_half_to_float(db);
            for (int l = 0; l < 32; l++)
                q[l] = (int16_t)(d > 0.0f ? qclamp(x[l] / d, lo - off, hi - off) + off : off);
        }
        rc = oq_pack(type, 1, q, s, m, &db, &dmb, out + i * bb);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Importance-weighted quantizer (the imatrix objective)                    */
/* ------------------------------------------------------------------------ */

/* [HG] 11.3 "I-quants and the importance matrix": plain quantization
 * minimises sum_i (w_i - w^_i)^2; with an importance matrix the quantizer
 * minimises sum_i E[x_i^2] (w_i - w^_i)^2, E[x_i^2] being the mean squared
 * activation met by weight column i.  The page states the objective, not the
 * search; the reading adopted (every step fp32, every sum sequential in
 * index order, no fused multiply-add):
 *   per group (the 32-weight block of Q8_0 / Q5_0 / Q4_0, the 32-weight
 *   sub-block of Q4_K / Q5_K, the 16-weight group of Q6_K / Q3_K / Q2_K),
 *   start from the plain scheme's scale s0 (and min m0 for the types with a
 *   min); for k = 0..20 take s = s0 * f_k, f_k = (90 + k) / 100, round the
 *   codes with (s, m0), refit by weighted least squares (the scale alone,
 *   or scale and min jointly: the 2x2 normal equations, kept only when the
 *   determinant, the scale and the min are > 0, > 0 and >= 0), and keep the
 *   candidate of least weighted error (the first on ties).  The winning
 *   (s, m) replace the plain (s0, m0) and the block is assembled exactly as
 *   by oq_quantize (super-block scales, 6-bit / int8 fields, codes rounded
 *   with the stored values).  Last, both that block and the plain block are
 *   decoded and their weighted errors compared (per-group sums, then the
 *   sum over groups, both in order): the plain block is kept unless the
 *   weighted one is no worse.  Importances: fp32 [cols], finite and >= 0. */

/* Group layout per type: weights per group, symmetric or not, plain divisor
 * (symmetric: s0 = max|w| / div) or step count (with a min: s0 = (hi - lo) /
 * steps), code range. */
static void group_geometry(int type, int* G, int* sym, float* div, int* qlo, int* qhi) {
    switch (type) {
    case OQ_Q8_0: *G = 32; *sym = 1; *div = 127.0f; *qlo = -128; *qhi = 127; break;
    case OQ_Q5_0: *G = 32; *sym = 1; *div = 15.0f; *qlo = -16; *qhi = 15; break;
    case OQ_Q4_0: *G = 32; *sym = 1; *div = 7.0f; *qlo = -8; *qhi = 7; break;
    case OQ_Q6_K: *G = 16; *sym = 1; *div = 32.0f; *qlo = -32; *qhi = 31; break;
    case OQ_Q3_K: *G = 16; *sym = 1; *div = 4.0f; *qlo = -4; *qhi = 3; break;
    case OQ_Q4_K: *G = 32; *sym = 0; *div = 15.0f; *qlo = 0; *qhi = 15; break;
    case OQ_Q5_K: *G = 32; *sym = 0; *div = 31.0f; *qlo = 0; *qhi = 31; break;
    default:      *G = 16; *sym = 0; *div = 3.0f; *qlo = 0; *qhi = 3; break;   /* Q2_K */
    }
}

/* The search of one group: (s, m) out; m stays 0 for symmetric groups. */
static void imatrix_group(const float* x, const float* a, int G, int sym, float div, int qlo, int qhi,
                          float* s_out, float* m_out) {
    float s0, m0 = 0.0f;
    if (sym) {
        float amax = 0.0f;
        for (int l = 0; l < G; l++) {
            float v = fabsf(x[l]);
            if (v > amax) amax = v;
        }
        s0 = amax / div;
    } else {
        float lo = 0.0f, hi = x[0];
        for (int l = 0; l < G; l++) {
            if (x[l] < lo) lo = x[l];
            if (x[l] > hi) hi = x[l];
        }
        s0 = (hi - lo) / div;
        m0 = -lo;
    }
    *s_out = s0;
    *m_out = m0;
    if (!(s0 > 0.0f)) return;
    float best = INFINITY;
    for (int k = 0; k <= 20; k++) {
        float s = s0 * ((float)(90 + k) / 100.0f);
        int q[32];
        for (int l = 0; l < G; l++) q[l] = sym ? qclamp(x[l] / s, qlo, qhi) : qclamp((x[l] + m0) / s, qlo, qhi);
        float ss, mm = 0.0f;
        if (sym) {
            float num = 0.0f, den = 0.0f;
            for (int l = 0; l < G; l++) {
                float aq = a[l] * (float)q[l];
                num = num + aq * x[l];
                den = den + aq * (float)q[l];
            }
            if (!(den > 0.0f)) continue;
            ss = num / den;
        } else {
            float Sa = 0.0f, Sq = 0.0f, Sqq = 0.0f, Sw = 0.0f, Swq = 0.0f;
            for (int l = 0; l < G; l++) {
                float aq = a[l] * (float)q[l];
                Sa = Sa + a[l];
                Sq = Sq + aq;
                Sqq = Sqq + aq * (float)q[l];
                Sw = Sw + a[l] * x[l];
                Swq = Swq + aq * x[l];
            }
            float det = Sqq * Sa - Sq * Sq;
            if (!(det > 0.0f)) continue;
            ss = (Swq * Sa - Sq * Sw) / det;
            mm = (Swq * Sq - Sqq * Sw) / det;
            if (!(ss > 0.0f) || !(mm >= 0.0f)) continue;
        }
        float e = 0.0f;
        for (int l = 0; l < G; l++) {
            float r = x[l] - (ss * (float)q[l] - mm);
            e = e + a[l] * (r * r);
        }
        if (e < best) {
            best = e;
            *s_out = ss;
            *m_out = mm;
        }
    }
}

/* Encode one block from per-group (s, m): the assembly of oq_quantize with
 * the group parameters given. */
static int encode_block(int type, const float* x, const float* sg, const float* mg, uint8_t* out) {
    int16_t q[256], s[16];
    uint8_t m[16];
    uint16_t db = 0, dmb = 0;
    memset(s, 0, sizeof s);
    memset(m, 0, sizeof m);
    if (type == OQ_Q4_K || type == OQ_Q5_K || type == OQ_Q2_K) {
        const int two = type == OQ_Q2_K;
        const int G = two ? 16 : 32, ng = two ? 16 : 8, top = type == OQ_Q5_K ? 31 : (two ? 3 : 15);
        const float fmax = two ? 15.0f : 63.0f;
        const int smax = two ? 15 : 63;
        float maxsc = 0.0f, maxm = 0.0f;
        for (int j = 0; j < ng; j++) {
            if (sg[j] > maxsc) maxsc = sg[j];
            if (mg[j] > maxm) maxm = mg[j];
        }
        db = oq_float_to_half(maxsc / fmax);
        dmb = oq_float_to_half(maxm / fmax);
        float d = oq_half_to_float(db), dmin = oq_half_to_float(dmb);
        for (int j = 0; j < ng; j++) {
            s[j] = (int16_t)(d > 0.0f ? qclamp(sg[j] / d, 0, smax) : 0);
            m[j] = (uint8_t)(dmin > 0.0f ? qclamp(mg[j] / dmin, 0, smax) : 0);
            float ds = d * (float)s[j];
            float dm = dmin * (float)m[j];
            for (int l = 0; l < G; l++)
                q[G * j + l] = (int16_t)(ds > 0.0f ? qclamp((x[G * j + l] + dm) / ds, 0, top) : 0);
        }
    } else if (type == OQ_Q6_K || type == OQ_Q3_K) {
        const int six = type == OQ_Q6_K;
        float maxs = 0.0f;
        for (int j = 0; j < 16; j++)
            if (sg[j] > maxs) maxs = sg[j];
        db = oq_float_to_half(maxs / (six ? 127.0f : 31.0f));
        float d = oq_half_to_float(db);
        for (int j = 0; j < 16; j++) {
            s[j] = (int16_t)(d > 0.0f ? qclamp(sg[j] / d, six ? -128 : -32, six ? 127 : 31) : 0);
            float ds = d * (float)s[j];
            for (int l = 0; l < 16; l++) {
                float v = x[16 * j + l];
                if (six) q[16 * j + l] = (int16_t)(ds != 0.0f ? qclamp(v / ds, -32, 31) + 32 : 32);
                else q[16 * j + l] = (int16_t)(ds != 0.0f ? qclamp(v / ds, -4, 3) : 0);
            }
        }
    } else {
        int off = (type == OQ_Q8_0) ? 0 : (type == OQ_Q5_0 ? 16 : 8);
        int lo = (type == OQ_Q8_0) ? -128 : 0;
        int hi = (type == OQ_Q8_0) ? 127 : (type == OQ_Q5_0 ? 31 : 15);
        db = oq_float_to_half(sg[0]);
        float d = oq_half_to_float(db);
        for (int l = 0; l < 32; l++)
            q[l] = (int16_t)(d > 0.0f ? qclamp(x[l] / d, lo - off, hi - off) + off : off);
    }
    return oq_pack(type, 1, q, s, m, &db, &dmb, out);
}

/* Weighted error of one encoded block against x: per-group sums in order,
 * then the sum over groups in order. */
static float block_error(int type, const uint8_t* blk, const float* x, const float* a) {
    float w[256];
    int G, sym, qlo, qhi;
    float div;
    group_geometry(type, &G, &sym, &div, &qlo, &qhi);
    dequant_block(type, blk, w);
    int be = oq_block_elems(type);
    float total = 0.0f;
    for (int g = 0; g < be / G; g++) {
        float e = 0.0f;
        for (int l = 0; l < G; l++) {
            float r = x[G * g + l] - w[G * g + l];
            e = e + a[G * g + l] * (r * r);
        }
        total = total + e;
    }
    return total;
}

int oq_quantize_imatrix(int type, const float* w, int64_t rows, int64_t cols, const float* imp, uint8_t* out) {
    int rc = check_shape(type, rows, cols);
    if (rc) return rc;
    int bb = oq_block_bytes(type), be = oq_block_elems(type);
    int G, sym, qlo, qhi;
    float div;
    group_geometry(type, &G, &sym, &div, &qlo, &qhi);
    int64_t nbr = cols / be;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t bi = 0; bi < nbr; bi++) {
            const float* x = w + r * cols + bi * be;
            const float* a = imp + bi * be;
            uint8_t* o = out + (r * nbr + bi) * bb;
            float sg[16], mg[16];
            for (int g = 0; g < be / G; g++) imatrix_group(x + G * g, a + G * g, G, sym, div, qlo, qhi, &sg[g], &mg[g]);
            uint8_t plain[256], mine[256];
            rc = oq_quantize(type, x, 1, be, plain);
            if (rc) return rc;
            rc = encode_block(type, x, sg, mg, mine);
            if (rc) return rc;
            float ep = block_error(type, plain, x, a), em = block_error(type, mine, x, a);
            memcpy(o, em <= ep ? mine : plain, (size_t)bb);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over a block-quantized KV cache                          */
/* ------------------------------------------------------------------------ */

/* [HG] 13.2 (KV-cache quantization at serve time): keys and values are
 * stored as q8_0 (or q4_0) blocks and read inside attention.  One query
 * token: for query head h (kv head g = h / (n_heads / n_kv), grouped-query
 * attention as the page describes), s_t = scale * sum_i q[h,i] K[t,g,i],
 * p = softmax(s) over t = 0..T-1, out[h,i] = sum_t p_t V[t,g,i].  K and V are
 * [T, n_kv, d] with each (t, g) row d/32 blocks of a 32-weight type; the
 * oracle dequantizes them exactly and does the rest in fp64 (softmax with the
 * maximum subtracted).  Sv[h,i] = sum_t p_t |V[t,g,i]| is returned for the
 * tolerance. */
int oq_attn_decode(int type, const float* q, const uint8_t* K, const uint8_t* V, int64_t T, int n_heads,
                   int n_kv, int d, float scale, double* out, double* Sv) {
    if (oq_block_elems(type) != 32 || d % 32 != 0 || n_kv <= 0 || n_heads % n_kv != 0 || T < 1) return -2;
    int bb = oq_block_bytes(type);
    int64_t rowb = (int64_t)(d / 32) * bb;
    int grp = n_heads / n_kv;
    float* k = (float*)malloc(sizeof(float) * (size_t)d);
    float* v = (float*)malloc(sizeof(float) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)T);
    if (!k || !v || !s) { free(k); free(v); free(s); return -3; }
    for (int h = 0; h < n_heads; h++) {
        int g = h / grp;
        double mx = -INFINITY;
        for (int64_t t = 0; t < T; t++) {
            const uint8_t* row = K + (t * n_kv + g) * rowb;
            for (int b = 0; b < d / 32; b++) dequant_block(type, row + b * bb, k + 32 * b);
            double acc = 0.0;
            for (int i = 0; i < d; i++) acc += (double)q[(int64_t)h * d + i] * (double)k[i];
            s[t] = (double)scale * acc;
            if (s[t] > mx) mx = s[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < T; t++) {
            s[t] = exp(s[t] - mx);
            l += s[t];
        }
        for (int i = 0; i < d; i++) {
            out[(int64_t)h * d + i] = 0.0;
            Sv[(int64_t)h * d + i] = 0.0;
        }
        for (int64_t t = 0; t < T; t++) {
            const uint8_t* row = V + (t * n_kv + g) * rowb;
            for (int b = 0; b < d / 32; b++) dequant_block(type, row + b * bb, v + 32 * b);
            double p = s[t] / l;
            for (int i = 0; i < d; i++) {
                out[(int64_t)h * d + i] += p * (double)v[i];
                Sv[(int64_t)h * d + i] += p * fabs((double)v[i]);
            }
        }
    }
    free(k);
    free(v);
    free(s);
    return 0;
}
