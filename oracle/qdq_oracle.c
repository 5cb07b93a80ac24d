/*
 * qdq_oracle.c -- plain, slow CPU oracle for block-quantised dequantisation and
 * the dequant-GEMV.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
 * CPU-baseline leg may call it; the library's compute path never does. It shares
 * no code, header or table with the CUDA path.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (-ffp-contract=off matters: on aarch64 gcc would otherwise fuse a*b-c into one
 * FMA and change the rounding the pages fix.)
 *
 * Every float operation below is one IEEE-754 binary32 operation in the order the
 * cited passage evaluates it. No blocking, fusion or reordering.
 *
 * Sources (page title, section):
 *   [S21]  "S21 The Capstone: picoLM, in Python", section 2 "K-quants"
 *          (Q4_K super-block diagram and dequantize_q4_K), section 3 (fused
 *          dequant + dot; the unfused reference path is dequantise-then-dot).
 *   [Q6K]  "PicoLM Q6_K quantisation bug" (block_q6_K struct; one int8 scale per
 *          16 weights; scale group = is + l/16; y = d * sc * q).
 *   [PETIT] "PETIT -- a tiny, CPU-first, quantized LLM inference engine",
 *          "What makes it fast & small" and "How the pieces match" (q8_0 = fp32
 *          scale + 32 int8; q4_0 = fp16 scale + 16 nibble bytes; weights stored
 *          out x in, one projection = one gemv).
 *
 * Pin status (what the tests hold each function to):
 *   fp16 -> fp32    pinned: all 65536 patterns vs numpy float16.
 *   Q4_K            pinned: hand-built blocks with closed-form values, the
 *                   12-byte scale/min field layout, mutations.
 *   Q6_K            pinned: struct offsets, one scale per 16 weights, the
 *                   scale[0]/scale[1] error ratio, closed forms. The placement
 *                   of each quant's 4 low bits in ql and 2 high bits in qh is
 *                   NOT printed on the pages: it follows the ggml layout (a
 *                   reading), and is "parity unpinned" against the pages.
 *   q8_0, q4_0      pinned: hand-built blocks with closed-form values. The q4_0
 *                   nibble order (low nibble = weight i, high = weight i+16) is
 *                   the workload definition's reading.
 *   Q5_0, Q5_1,     layouts not on the pages (ggml's, a reading): pinned by
 *   ggml q8_0, Q2_K hand-built blocks and mutations; Q2_K also by the page's 84
 *   Q5_K, Q3_K      bytes per 256 weights. "Parity unpinned" against the pages
 *                   for the bit placements.
 *   GEMV            pinned: exact rational sums on tiny inputs, unit-vector
 *                   columns (catches a transposed operand), closed forms.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_Q4_0 = 1, ORC_Q8_0 = 2, ORC_Q4_K = 3, ORC_Q6_K = 4, ORC_Q5_0 = 5, ORC_Q5_1 = 6, ORC_Q8_0G = 7,
       ORC_Q2_K = 8, ORC_Q5_K = 9, ORC_Q3_K = 10 };

/* ---- IEEE-754 binary16 -> binary32, from the format definition ---------------
 * sign s (1 bit), exponent e (5 bits, bias 15), fraction f (10 bits):
 *   e == 0        : (-1)^s * f * 2^-24          (zero, subnormal)
 *   0 < e < 31    : (-1)^s * (1024 + f) * 2^(e-25)
 *   e == 31       : f == 0 ? (-1)^s * inf : NaN
 * Every binary16 value is exactly representable in binary32.                    */
float orc_fp16_to_fp32(uint16_t h) {
    unsigned s = (h >> 15) & 1u, e = (h >> 10) & 31u, f = h & 1023u;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? (double)NAN : (double)INFINITY;
    else
        v = ldexp((double)(1024u + f), (int)e - 25);
    return (float)(s ? -v : v);
}

static float rd_fp16(const uint8_t *p) { return orc_fp16_to_fp32((uint16_t)(p[0] | (p[1] << 8))); }

/* ---- Q4_K: 144 bytes -> 256 weights [S21 section 2] ----------------------------
 * bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 (p[0..11] below) eight 6-bit scales and
 * eight 6-bit mins, one pair per 32-weight sub-block, bit-packed (the page's
 * super-block diagram: 12 bytes of packed 6-bit scales and mins; fields 4-7
 * straddle byte boundaries).
 * Where bit b of field j of kind k (k = 0: scale, 1: min) lives in p:
 *   fields 0-3 sit whole in the low six bits of one byte: scales in bytes 0-3,
 *     mins in bytes 4-7 (byte 4k + j, bit b);
 *   fields 4-7 keep their four low bits in byte j+4, scales in its low nibble
 *     and mins in its high nibble (bit 4k + b), and their two top bits in bits
 *     6-7 of the byte that holds field j-4 of the same kind (byte 4k + j - 4,
 *     bit 6 + b - 4).
 * The value is assembled one bit at a time from those positions.               */
static void q4k_field_bit(int k, int j, int b, int *byte, int *bit) {
    if (j < 4) {
        *byte = 4 * k + j;
        *bit = b;
    } else if (b < 4) {
        *byte = j + 4;
        *bit = 4 * k + b;
    } else {
        *byte = 4 * k + (j - 4);
        *bit = 6 + (b - 4);
    }
}

void orc_q4k_scale_min(const uint8_t *p, int j, int *sc, int *mn) {
    int v[2] = {0, 0};
    for (int k = 0; k < 2; ++k)
        for (int b = 0; b < 6; ++b) {
            int byte, bit;
            q4k_field_bit(k, j, b, &byte, &bit);
            v[k] |= ((p[byte] >> bit) & 1) << b;
        }
    *sc = v[0];
    *mn = v[1];
}

/* The nibble bytes form four chunks of 32 bytes. In chunk c the low nibbles are
 * weights 64c..64c+31 (sub-block 2c) and the high nibbles are weights
 * 64c+32..64c+63 (sub-block 2c+1). Value, evaluated left to right as the page's
 * NumPy expression does: (d * sc) * q - (dmin * mn).                            */
void orc_dequant_q4_K_block(const uint8_t *blk, float *out) {
    float d = rd_fp16(blk), dmin = rd_fp16(blk + 2);
    const uint8_t *p = blk + 4, *qs = blk + 16;
    for (int e = 0; e < 256; ++e) {
        int c = e / 64, i = e % 64;
        int s = 2 * c + (i >= 32);
        int q = (i < 32) ? (qs[32 * c + i] & 15) : (qs[32 * c + i - 32] >> 4);
        int sc, mn;
        orc_q4k_scale_min(p, s, &sc, &mn);
        float a = d * (float)sc;
        a = a * (float)q;
        float b = dmin * (float)mn;
        out[e] = a - b;
    }
}

/* ---- Q6_K: 210 bytes -> 256 weights [Q6K] -------------------------------------
 * struct { uint8 ql[128]; uint8 qh[64]; int8 scales[16]; fp16 d; }.
 * Each quant has six bits: four in ql, two in qh (placement: ggml layout, a
 * reading -- see the header). Element e = 128h + 32k + l (h = half, k = 0..3,
 * l = 0..31):
 *   low  = ql[64h + 32(k & 1) + l], low nibble for k < 2, high nibble for k >= 2
 *   high = (qh[32h + l] >> 2k) & 3
 *   q    = (low | high << 4) - 32
 * One scale per 16 weights: element e uses scales[e / 16]. This is the fixed
 * rule "is + l/16" of the page: with is = 8h, y[l], y[l+32], y[l+64], y[l+96]
 * take sc[is + l/16 + 0, 2, 4, 6].
 * Value, left to right as the page's C: (d * sc) * q.                           */
void orc_dequant_q6_K_block(const uint8_t *blk, float *out) {
    const uint8_t *ql = blk, *qh = blk + 128;
    const int8_t *scales = (const int8_t *)(blk + 192);
    float d = rd_fp16(blk + 208);
    for (int e = 0; e < 256; ++e) {
        int h = e / 128, k = (e % 128) / 32, l = e % 32;
        int lb = ql[64 * h + 32 * (k & 1) + l];
        int low = (k < 2) ? (lb & 15) : (lb >> 4);
        int high = (qh[32 * h + l] >> (2 * k)) & 3;
        int q = (low | (high << 4)) - 32;
        float a = d * (float)scales[e / 16];
        out[e] = a * (float)q;
    }
}

/* ---- PETIT q8_0: 36 bytes -> 32 weights [PETIT] --------------------------------
 * fp32 scale d, then 32 int8 q. w = d * q (one rounding).                       */
void orc_dequant_q8_0_block(const uint8_t *blk, float *out) {
    float d;
    memcpy(&d, blk, 4); /* little-endian host; the format is little-endian */
    const int8_t *q = (const int8_t *)(blk + 4);
    for (int i = 0; i < 32; ++i) out[i] = d * (float)q[i];
}

/* ---- PETIT q4_0: 18 bytes -> 32 weights [PETIT] --------------------------------
 * fp16 scale d, then 16 bytes; byte i holds weight i in its low nibble and
 * weight i+16 in its high nibble; w = (q - 8) * d (one rounding).               */
void orc_dequant_q4_0_block(const uint8_t *blk, float *out) {
    float d = rd_fp16(blk);
    const uint8_t *qs = blk + 2;
    for (int i = 0; i < 32; ++i) {
        int q = (i < 16) ? (qs[i] & 15) : (qs[i - 16] >> 4);
        out[i] = (float)(q - 8) * d;
    }
}

/* ---- More GGUF formats [S21 section 2: "eight formats", Q2_K 84 bytes per 256;
 * the layouts themselves are not on the pages] -----------------------------------
 * These follow the published ggml block layouts (a reading; pinned against the
 * pages only by Q2_K's 84 bytes per 256 weights, and by hand-built blocks).
 *
 * Q5_0: 22 bytes -> 32 weights: fp16 d; qh, four bytes read as a little-endian
 * 32-bit word whose bit i is the fifth bit of weight i; 16 bytes qs, byte i
 * holding weight i in its low nibble and weight i+16 in its high nibble.
 * q = nibble | bit << 4 (0..31); w = (q - 16) * d (one rounding).               */
static int q5_quant(const uint8_t *qh4, const uint8_t *qs, int i) {
    uint32_t qh = (uint32_t)qh4[0] | ((uint32_t)qh4[1] << 8) | ((uint32_t)qh4[2] << 16) | ((uint32_t)qh4[3] << 24);
    int nib = (i < 16) ? (qs[i] & 15) : (qs[i - 16] >> 4);
    return nib | (int)(((qh >> i) & 1u) << 4);
}

void orc_dequant_q5_0_block(const uint8_t *blk, float *out) {
    float d = rd_fp16(blk);
    for (int i = 0; i < 32; ++i) out[i] = (float)(q5_quant(blk + 2, blk + 6, i) - 16) * d;
}

/* Q5_1: 24 bytes: fp16 d, fp16 m, qh, qs as Q5_0; w = q * d + m (q * d is exact
 * in binary32, so this is one rounding).                                         */
void orc_dequant_q5_1_block(const uint8_t *blk, float *out) {
    float d = rd_fp16(blk), m = rd_fp16(blk + 2);
    for (int i = 0; i < 32; ++i) {
        float a = (float)q5_quant(blk + 4, blk + 8, i) * d;
        out[i] = a + m;
    }
}

/* ggml q8_0: 34 bytes: fp16 d, 32 int8 q; w = q * d. (PETIT's q8_0 has an fp32
 * scale instead.)                                                                */
void orc_dequant_q8_0g_block(const uint8_t *blk, float *out) {
    float d = rd_fp16(blk);
    const int8_t *q = (const int8_t *)(blk + 2);
    for (int i = 0; i < 32; ++i) out[i] = (float)q[i] * d;
}

/* Q2_K: 84 bytes -> 256 weights: 16 scale bytes (low nibble: scale, high nibble:
 * min, one pair per 16 weights), 64 bytes of 2-bit quants, fp16 d, fp16 dmin.
 * Element e = 128n + 32j + l (n = half, j = 0..3, l = 0..31): q = bits 2j..2j+1
 * of qs[32n + l]; its pair is scales[8n + 2j + l/16].
 * Value, left to right: (d * sc) * q - (dmin * mn).                              */
void orc_dequant_q2_K_block(const uint8_t *blk, float *out) {
    const uint8_t *scales = blk, *qs = blk + 16;
    float d = rd_fp16(blk + 80), dmin = rd_fp16(blk + 82);
    for (int e = 0; e < 256; ++e) {
        int n = e / 128, j = (e % 128) / 32, l = e % 32;
        int q = (qs[32 * n + l] >> (2 * j)) & 3;
        int sm = scales[8 * n + 2 * j + l / 16];
        float a = d * (float)(sm & 15);
        a = a * (float)q;
        float b = dmin * (float)(sm >> 4);
        out[e] = a - b;
    }
}

/* Q5_K: 176 bytes -> 256 weights: fp16 d, fp16 dmin, the 12-byte scale/min
 * field of Q4_K (same packing), qh[32], qs[128]. Element e = 64c + 32h + l
 * (c = 0..3, h = 0 low / 1 high, l = 0..31): its four low bits are the low (h =
 * 0) or high (h = 1) nibble of qs[32c + l], its fifth bit is bit 2c + h of
 * qh[l]; sub-block 2c + h. Value, left to right: (d * sc) * q - (dmin * mn),
 * q in 0..31 (d * sc * q is exact: 11 + 6 + 5 bits).                           */
void orc_dequant_q5_K_block(const uint8_t *blk, float *out) {
    const float dmin = rd_fp16(blk + 2), d = rd_fp16(blk);
    const uint8_t *fields = blk + 4, *qh = blk + 16, *qs = blk + 48;
    for (int e = 0; e < 256; ++e) {
        int c = e / 64, h = (e % 64) / 32, l = e % 32, sb = 2 * c + h;
        int sc, mn;
        orc_q4k_scale_min(fields, sb, &sc, &mn);
        int nib = h ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
        int q = nib | (((qh[l] >> sb) & 1) << 4);
        float a = d * (float)sc;
        a = a * (float)q;
        float b = dmin * (float)mn;
        out[e] = a - b;
    }
}

/* Q3_K: 110 bytes -> 256 weights: hmask[32], qs[64] of 2-bit quants, 12 bytes of
 * sixteen 6-bit scales, fp16 d at byte 108. Element e = 128n + 32j + l (n = half,
 * j = 0..3, l = 0..31): q = (bits 2j..2j+1 of qs[32n + l]) - 4 when bit 4n + j of
 * hmask[l] is clear (else - 0), so q in -4..3; sub-block s = 8n + 2j + l/16 of
 * 16 weights. Scale s: low four bits in byte s (s < 8, low nibble) or byte s - 8
 * (s >= 8, high nibble) of the field, top two bits at bit 2 (s / 4) of byte
 * 8 + s % 4; the scale is that 6-bit value minus 32. Value: (d * scale) * q,
 * exact (11 + 6 + 3 bits).                                                      */
static int q3k_scale(const uint8_t *f, int s) {
    int low = s < 8 ? (f[s] & 15) : (f[s - 8] >> 4);
    int high = (f[8 + s % 4] >> (2 * (s / 4))) & 3;
    return (low | (high << 4)) - 32;
}

void orc_dequant_q3_K_block(const uint8_t *blk, float *out) {
    const uint8_t *hmask = blk, *qs = blk + 32, *f = blk + 96;
    float d = rd_fp16(blk + 108);
    for (int e = 0; e < 256; ++e) {
        int n = e / 128, j = (e % 128) / 32, l = e % 32;
        int low2 = (qs[32 * n + l] >> (2 * j)) & 3;
        int q = ((hmask[l] >> (4 * n + j)) & 1) ? low2 : low2 - 4;
        float a = d * (float)q3k_scale(f, 8 * n + 2 * j + l / 16);
        out[e] = a * (float)q;
    }
}

int orc_block_bytes(int type) {
    switch (type) {
    case ORC_Q4_0: return 18;
    case ORC_Q8_0: return 36;
    case ORC_Q4_K: return 144;
    case ORC_Q6_K: return 210;
    case ORC_Q5_0: return 22;
    case ORC_Q5_1: return 24;
    case ORC_Q8_0G: return 34;
    case ORC_Q2_K: return 84;
    case ORC_Q5_K: return 176;
    case ORC_Q3_K: return 110;
    default: return -1;
    }
}

int orc_block_weights(int type) {
    switch (type) {
    case ORC_Q4_0: case ORC_Q8_0: case ORC_Q5_0: case ORC_Q5_1: case ORC_Q8_0G: return 32;
    case ORC_Q4_K: case ORC_Q6_K: case ORC_Q2_K: case ORC_Q5_K: case ORC_Q3_K: return 256;
    default: return -1;
    }
}

/* Dequantise n weights (n a multiple of the block size). Returns 0, or -1 on a
 * bad type or size.                                                            */
int orc_dequant(int type, const uint8_t *blocks, int64_t n, float *out) {
    int bw = orc_block_weights(type), bb = orc_block_bytes(type);
    if (bw < 0 || n < 0 || n % bw) return -1;
    for (int64_t b = 0; b < n / bw; ++b) {
        const uint8_t *blk = blocks + b * bb;
        float *o = out + b * bw;
        switch (type) {
        case ORC_Q4_K: orc_dequant_q4_K_block(blk, o); break;
        case ORC_Q6_K: orc_dequant_q6_K_block(blk, o); break;
        case ORC_Q8_0: orc_dequant_q8_0_block(blk, o); break;
        case ORC_Q4_0: orc_dequant_q4_0_block(blk, o); break;
        case ORC_Q5_0: orc_dequant_q5_0_block(blk, o); break;
        case ORC_Q5_1: orc_dequant_q5_1_block(blk, o); break;
        case ORC_Q8_0G: orc_dequant_q8_0g_block(blk, o); break;
        case ORC_Q2_K: orc_dequant_q2_K_block(blk, o); break;
        case ORC_Q5_K: orc_dequant_q5_K_block(blk, o); break;
        case ORC_Q3_K: orc_dequant_q3_K_block(blk, o); break;
        }
    }
    return 0;
}

/* ---- GEMV: the unfused definition [S21 section 3; PETIT] ----------------------
 * W is rows x cols (out x in), row-major, each row cols/QK whole blocks.
 * x is [batch][cols], y and S are [batch][rows]. For each row: dequantise the row
 * to fp32 exactly as above, then in double precision
 *   y[b][r] = sum_c w[r][c] * x[b][c]      S[b][r] = sum_c |w[r][c] * x[b][c]|
 * summed in column order. Each double product of two floats is exact.
 * `row_buf` holds cols floats. Rows [r0, r1) only, so callers can sample.      */
int orc_gemv_rows(int type, const uint8_t *W, int64_t rows, int64_t cols, const float *x,
                  int batch, int64_t r0, int64_t r1, double *y, double *S, float *row_buf) {
    int bw = orc_block_weights(type), bb = orc_block_bytes(type);
    if (bw < 0 || cols % bw || rows < 0 || batch < 1 || r0 < 0 || r1 > rows || r0 > r1) return -1;
    int64_t rbytes = (cols / bw) * bb;
    for (int64_t r = r0; r < r1; ++r) {
        if (orc_dequant(type, W + r * rbytes, cols, row_buf)) return -1;
        for (int b = 0; b < batch; ++b) {
            const float *xb = x + (int64_t)b * cols;
            double acc = 0.0, sabs = 0.0;
            for (int64_t c = 0; c < cols; ++c) {
                double p = (double)row_buf[c] * (double)xb[c];
                acc += p;
                sabs += fabs(p);
            }
            y[(int64_t)b * rows + r] = acc;
            S[(int64_t)b * rows + r] = sabs;
        }
    }
    return 0;
}
