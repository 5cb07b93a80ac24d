// qdq_decode.cuh -- block-format field decoders, shared by the standalone
// dequantisation kernel and the fused GEMV.
//
// Layouts:
//   Q4_K ("S21 The Capstone: picoLM, in Python", section 2): 144 bytes = fp16 d,
//        fp16 dmin, 12 bytes p[0..11] of 6-bit scale/min fields, 128 nibble bytes
//        in four 32-byte chunks. Sub-block j (32 weights): j < 4 keeps its scale
//        in the low six bits of p[j] and its min in the low six bits of p[j+4];
//        j >= 4 keeps the low four bits of both in p[j+4] (scale low nibble, min
//        high nibble) and the top two bits in bits 6-7 of p[j-4] (scale) and
//        p[j] (min). Chunk c holds sub-block 2c in its low nibbles and 2c+1 in
//        its high nibbles.
//   Q6_K ("PicoLM Q6_K quantisation bug", block_q6_K): ql[128], qh[64],
//        int8 scales[16] (one per 16 weights: element e uses scales[e/16]), fp16
//        d at byte 208. Element e = 128h + 32k + l has low four bits in
//        ql[64h + 32(k&1) + l] (low nibble for k < 2, high for k >= 2) and top two
//        bits at bit 2k of qh[32h + l] (the ggml placement); q = q6 - 32.
//   PETIT q8_0 / q4_0 ("PETIT", How the pieces match): fp32 d + 32 int8, and
//        fp16 d + 16 bytes whose low nibbles are weights 0-15 and high nibbles
//        weights 16-31.
#pragma once
#include <cstdint>

#include "qdq_device.cuh"

namespace qdq {

// ---- Q4_K -------------------------------------------------------------------------
// Header words of a Q4_K block: H0 = d | dmin << 16, H1 = p[0..3], H2 = p[4..7],
// H3 = p[8..11] (little-endian bytes).
// Returns the 6-bit scales of sub-blocks 2c and 2c+1 in bytes 0 and 1 of *sc and
// their mins in bytes 0 and 1 of *mn.
QDQ_DEV void q4k_pair_fields(uint32_t H1, uint32_t H2, uint32_t H3, int c, uint32_t *sc,
                             uint32_t *mn) {
    // Branch-free over c, so the four chunk lanes of a super-block do not diverge.
    const uint32_t sh = 16u * (uint32_t)(c & 1);
    const uint32_t upper = (uint32_t)(c >> 1);  // 0: sub-blocks 0..3, 1: sub-blocks 4..7
    const uint32_t top = 2u * upper;            // the top two bits sit at bits 4-5 or 6-7
    const uint32_t a = (upper ? H3 : H1) >> sh;
    const uint32_t b = (upper ? (H3 >> 4) : H2) >> sh;
    *sc = (a & 0x0F0Fu) | (((H1 >> sh) >> top) & 0x3030u);
    *mn = (b & 0x0F0Fu) | (((H2 >> sh) >> top) & 0x3030u);
}

// Recentering of a Q4_K sub-block for the factored dot product. With s = d sc and
// m = dmin mn (both exact in fp32: an 11-bit fp16 significand times a 6-bit field),
// every weight is w = s q - m, q in 0..15. Summing s (q - rho) x - (m - s rho) x over
// the sub-block, with rho the integer in [0, 15] nearest to m / s, keeps both
// factored terms within a small multiple of sum |w x|: |m - s rho| <= |s| / 2, and
// m - s rho is exact (Sterbenz) whenever rho is not clamped. Without it, a sub-block
// whose weights nearly cancel (s q close to m) would lose the result to rounding.
// Returns rho; *m_rest = m - s rho. Degenerate s (zero, non-finite ratio) gives
// rho = 0 or 15 and the plain form.
QDQ_DEV float q4k_center(float s, float m, float *m_rest) {
    const float rho = fminf(fmaxf(rintf(__fdividef(m, s)), 0.0f), 15.0f);
    *m_rest = fmaf(-s, rho, m);
    return rho;
}

// ---- Q6_K -------------------------------------------------------------------------
// Given the ql word holding bytes l..l+3 of the run used by k (run k&1) and the qh
// word holding bytes l..l+3 of qh's half, returns the four 6-bit quants q6 of
// elements 128h + 32k + l .. +3 as the bytes of one word.
QDQ_DEV uint32_t q6k_quant_bytes(uint32_t ql, uint32_t qh, int k) {
    const uint32_t low = (k < 2) ? (ql & 0x0F0F0F0Fu) : ((ql >> 4) & 0x0F0F0F0Fu);
    uint32_t high;
    switch (k) {
        case 0: high = qh << 4; break;
        case 1: high = qh << 2; break;
        case 2: high = qh; break;
        default: high = qh >> 2; break;
    }
    uint32_t q6;  // low | (high & 0x30303030) as one LOP3
    asm("lop3.b32 %0, %1, %2, %3, 0xF8;" : "=r"(q6) : "r"(low), "r"(high), "n"(0x30303030));
    return q6;
}

// ---- exact per-weight values (for the dequantisation kernel) ---------------------
// No fused multiply-add: every product and difference is rounded once, in the
// pages' order.
QDQ_DEV float q4k_weight(float d, float dmin, uint32_t sc, uint32_t mn, uint32_t q) {
    return __fsub_rn(__fmul_rn(__fmul_rn(d, (float)sc), (float)q), __fmul_rn(dmin, (float)mn));
}
QDQ_DEV float q6k_weight(float d, int sc, int q6) { return __fmul_rn(__fmul_rn(d, (float)sc), (float)(q6 - 32)); }
QDQ_DEV float q8_0_weight(float d, int q) { return __fmul_rn(d, (float)q); }
QDQ_DEV float q4_0_weight(float d, int q) { return __fmul_rn((float)(q - 8), d); }

// ---- integer -> float by exponent-field construction (for the fused GEMV) --------
// For an integer v < 2^23 placed in the low mantissa bits, the float with bits
// 0x4B000000 | v equals 2^23 + v exactly; subtracting 2^23 (or 2^23 + offset) in
// fp32 gives v (or v - offset) exactly. A nibble can stay at its bit position p
// (value q * 2^p) as long as p + 4 <= 23; the matching x is pre-scaled by 2^-p.
constexpr uint32_t kMagic = 0x4B000000u;
constexpr float kTwo23 = 8388608.0f;

// One byte of `w` (selector j) as the float 2^23 + byte, in one byte permute.
template <int J>
QDQ_DEV uint32_t byte_to_magic(uint32_t w) {
    return __byte_perm(w, kMagic, (uint32_t)J | 0x7440u);
}


// ---- four consecutive weights of one block, exactly (shared by the standalone
// dequantisation kernel and the tensor-core path) -------------------------------
QDQ_DEV uint32_t ldg_u16(const uint8_t *p) { return (uint32_t)__ldg((const unsigned short *)p); }
QDQ_DEV uint32_t ldg_u32(const uint8_t *p) { return __ldg((const unsigned int *)p); }
// 4 bytes at a 2-byte-aligned address
QDQ_DEV uint32_t ldg_u32_a2(const uint8_t *p) { return ldg_u16(p) | (ldg_u16(p + 2) << 16); }

// Block geometry of every format the decoder knows.
__host__ __device__ constexpr int fmt_bytes(int t) {
    return t == QDQ_Q4_K ? 144 : t == QDQ_Q6_K ? 210 : t == QDQ_Q8_0 ? 36 : t == QDQ_Q4_0 ? 18 : t == QDQ_Q5_0 ? 22
           : t == QDQ_Q5_1 ? 24 : t == QDQ_Q8_0_GGML ? 34 : t == QDQ_Q2_K ? 84 : t == QDQ_Q5_K ? 176
           : t == QDQ_Q3_K ? 110 : 0;
}
__host__ __device__ constexpr int fmt_weights(int t) {
    return (t == QDQ_Q4_K || t == QDQ_Q6_K || t == QDQ_Q2_K || t == QDQ_Q5_K || t == QDQ_Q3_K) ? 256 : 32;
}

// Weights e0 .. e0+3 (e0 a multiple of 4) of the block at `blk`.
template <int TYPE>
QDQ_DEV float4 decode4(const uint8_t *blk, int e0) {
    float4 v;
    if constexpr (TYPE == QDQ_Q4_K) {  // blk 16-byte aligned
        const uint4 H = __ldg((const uint4 *)blk);
        const int c = e0 >> 6, i = e0 & 63;
        const bool high = i >= 32;
        uint32_t sc2, mn2;
        q4k_pair_fields(H.y, H.z, H.w, c, &sc2, &mn2);
        const uint32_t sc = high ? (sc2 >> 8) : (sc2 & 0xFF);
        const uint32_t mn = high ? (mn2 >> 8) : (mn2 & 0xFF);
        const float d = half_bits_to_float(H.x & 0xFFFF), dmin = half_bits_to_float(H.x >> 16);
        uint32_t q = ldg_u32(blk + 16 + 32 * c + (i & 31));
        if (high) q >>= 4;
        v.x = q4k_weight(d, dmin, sc, mn, q & 15);
        v.y = q4k_weight(d, dmin, sc, mn, (q >> 8) & 15);
        v.z = q4k_weight(d, dmin, sc, mn, (q >> 16) & 15);
        v.w = q4k_weight(d, dmin, sc, mn, (q >> 24) & 15);
    } else if constexpr (TYPE == QDQ_Q6_K) {  // blk 2-byte aligned
        const int h = e0 >> 7, k = (e0 >> 5) & 3, l = e0 & 31;
        const uint32_t ql = ldg_u32_a2(blk + 64 * h + 32 * (k & 1) + l);
        const uint32_t qh = ldg_u32_a2(blk + 128 + 32 * h + l);
        const int sc = (int)(int8_t)__ldg(blk + 192 + (e0 >> 4));
        const float d = half_bits_to_float(ldg_u16(blk + 208));
        const uint32_t q6 = q6k_quant_bytes(ql, qh, k);
        v.x = q6k_weight(d, sc, (int)(q6 & 0xFF));
        v.y = q6k_weight(d, sc, (int)((q6 >> 8) & 0xFF));
        v.z = q6k_weight(d, sc, (int)((q6 >> 16) & 0xFF));
        v.w = q6k_weight(d, sc, (int)(q6 >> 24));
    } else if constexpr (TYPE == QDQ_Q8_0) {  // blk 4-byte aligned
        const float d = __uint_as_float(ldg_u32(blk));
        const uint32_t q = ldg_u32(blk + 4 + e0);
        v.x = q8_0_weight(d, (int)(int8_t)(q & 0xFF));
        v.y = q8_0_weight(d, (int)(int8_t)((q >> 8) & 0xFF));
        v.z = q8_0_weight(d, (int)(int8_t)((q >> 16) & 0xFF));
        v.w = q8_0_weight(d, (int)(int8_t)(q >> 24));
    } else if constexpr (TYPE == QDQ_Q5_0 || TYPE == QDQ_Q5_1) {  // blk 2-byte aligned
        // q = nibble | fifth bit << 4; Q5_0: (q - 16) * d; Q5_1: q * d + m (q * d exact)
        constexpr int kQh = TYPE == QDQ_Q5_0 ? 2 : 4;
        const float d = half_bits_to_float(ldg_u16(blk));
        const float m = TYPE == QDQ_Q5_1 ? half_bits_to_float(ldg_u16(blk + 2)) : 0.0f;
        const uint32_t qh = ldg_u32_a2(blk + kQh) >> e0;
        uint32_t q = ldg_u32_a2(blk + kQh + 4 + (e0 & 15));
        if (e0 >= 16) q >>= 4;
        float w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int qq = (int)(((q >> (8 * k)) & 15) | (((qh >> k) & 1) << 4));
            if constexpr (TYPE == QDQ_Q5_0)
                w[k] = __fmul_rn((float)(qq - 16), d);
            else
                w[k] = __fadd_rn(__fmul_rn((float)qq, d), m);
        }
        v = make_float4(w[0], w[1], w[2], w[3]);
    } else if constexpr (TYPE == QDQ_Q8_0_GGML) {  // blk 2-byte aligned
        const float d = half_bits_to_float(ldg_u16(blk));
        const uint32_t q = ldg_u32_a2(blk + 2 + e0);
        v.x = __fmul_rn((float)(int)(int8_t)(q & 0xFF), d);
        v.y = __fmul_rn((float)(int)(int8_t)((q >> 8) & 0xFF), d);
        v.z = __fmul_rn((float)(int)(int8_t)((q >> 16) & 0xFF), d);
        v.w = __fmul_rn((float)(int)(int8_t)(q >> 24), d);
    } else if constexpr (TYPE == QDQ_Q2_K) {  // blk 4-byte aligned
        // weight 128n + 32j + l: bits 2j..2j+1 of qs[32n + l], pair 8n + 2j + l/16;
        // (d * sc) * q - (dmin * mn), evaluated left to right
        const int n = e0 >> 7, j = (e0 >> 5) & 3, l = e0 & 31;
        const uint32_t q = ldg_u32(blk + 16 + 32 * n + l) >> (2 * j);
        const uint32_t sm = __ldg(blk + 8 * n + 2 * j + (l >> 4));
        const float dl = __fmul_rn(half_bits_to_float(ldg_u16(blk + 80)), (float)(sm & 15));
        const float ml = __fmul_rn(half_bits_to_float(ldg_u16(blk + 82)), (float)(sm >> 4));
        v.x = __fsub_rn(__fmul_rn(dl, (float)(q & 3)), ml);
        v.y = __fsub_rn(__fmul_rn(dl, (float)((q >> 8) & 3)), ml);
        v.z = __fsub_rn(__fmul_rn(dl, (float)((q >> 16) & 3)), ml);
        v.w = __fsub_rn(__fmul_rn(dl, (float)((q >> 24) & 3)), ml);
    } else if constexpr (TYPE == QDQ_Q5_K) {  // blk 16-byte aligned
        // the Q4_K header; weight 64c + 32h + l: nibble h of qs[32c + l], fifth
        // bit at bit 2c + h of qh[l]; (d * sc) * q - (dmin * mn)
        const uint4 H = __ldg((const uint4 *)blk);
        const int c = e0 >> 6, h = (e0 >> 5) & 1, l = e0 & 31;
        uint32_t sc2, mn2;
        q4k_pair_fields(H.y, H.z, H.w, c, &sc2, &mn2);
        const uint32_t sc = h ? (sc2 >> 8) : (sc2 & 0xFF);
        const uint32_t mn = h ? (mn2 >> 8) : (mn2 & 0xFF);
        const float d = half_bits_to_float(H.x & 0xFFFF), dmin = half_bits_to_float(H.x >> 16);
        const uint32_t q = ldg_u32(blk + 48 + 32 * c + l) >> (4 * h);
        const uint32_t qh = ldg_u32(blk + 16 + l) >> (2 * c + h);
        v.x = q4k_weight(d, dmin, sc, mn, (q & 15) | ((qh & 1) << 4));
        v.y = q4k_weight(d, dmin, sc, mn, ((q >> 8) & 15) | (((qh >> 8) & 1) << 4));
        v.z = q4k_weight(d, dmin, sc, mn, ((q >> 16) & 15) | (((qh >> 16) & 1) << 4));
        v.w = q4k_weight(d, dmin, sc, mn, ((q >> 24) & 15) | (((qh >> 24) & 1) << 4));
    } else if constexpr (TYPE == QDQ_Q3_K) {  // blk 2-byte aligned
        // weight 128n + 32j + l: bits 2j..2j+1 of qs[32n + l] minus 4 unless bit
        // 4n + j of hmask[l] is set; scale s = 8n + 2j + l/16 (6 bits, minus 32);
        // (d * scale) * q, exact
        const int n = e0 >> 7, j = (e0 >> 5) & 3, l = e0 & 31, s = 8 * n + 2 * j + (l >> 4);
        const uint32_t q = ldg_u32_a2(blk + 32 + 32 * n + l) >> (2 * j);
        const uint32_t hm = ldg_u32_a2(blk + l) >> (4 * n + j);
        const uint32_t lo = s < 8 ? (__ldg(blk + 96 + s) & 15u) : (__ldg(blk + 96 + s - 8) >> 4);
        const uint32_t hi = (__ldg(blk + 104 + (s & 3)) >> (2 * (s >> 2))) & 3u;
        const float dl = __fmul_rn(half_bits_to_float(ldg_u16(blk + 108)), (float)((int)(lo | (hi << 4)) - 32));
        float w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q2 = (int)((q >> (8 * k)) & 3u);
            w[k] = __fmul_rn(dl, (float)(((hm >> (8 * k)) & 1u) ? q2 : q2 - 4));
        }
        v = make_float4(w[0], w[1], w[2], w[3]);
    } else {  // QDQ_Q4_0, blk 2-byte aligned
        const float d = half_bits_to_float(ldg_u16(blk));
        uint32_t q = ldg_u32_a2(blk + 2 + (e0 & 15));
        if (e0 >= 16) q >>= 4;
        v.x = q4_0_weight(d, (int)(q & 15));
        v.y = q4_0_weight(d, (int)((q >> 8) & 15));
        v.z = q4_0_weight(d, (int)((q >> 16) & 15));
        v.w = q4_0_weight(d, (int)((q >> 24) & 15));
    }
    return v;
}

}  // namespace qdq
