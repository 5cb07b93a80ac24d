// qdq_stream_common.cuh -- pieces of the streaming (CUDA-core) GEMV kernel that
// the host-side plan packing shares with it: the packed kernel arguments, the
// format constants, the bulk-copy helper and the batch-1 dequant-dot units.
//
// "S21 The Capstone: picoLM, in Python", section 3 (fused dequant + dot product:
// the quantised bytes are decoded in registers and multiplied straight into the
// accumulator); "PETIT" (gemv_q8 / gemv_q4 over rows of 32-weight blocks).
#pragma once
#include <cstdint>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {
struct DevDesc {
    const uint8_t *W;
    const float *x;
    float *y;
    int64_t rows;
    int32_t cols;
    int32_t type;
    int32_t rb;     // bytes per row
    int32_t pad0;   // keeps the fields below at the offsets the kernel's register allocation was tuned with
    int32_t kinds;  // bit k: the level's x needs swizzled copy kind k (0 plain, 1 Q4_K-scaled, 2 q4_0-scaled)
    int32_t pad1;
};

template <int MAXD, int MAXL>
struct StreamArgs {
    int32_t ndesc, nlevels, batch, pad;
    unsigned *counters;
    unsigned long long *trace;  // QDQ_TRACE builds only: per-CTA phase timestamps
    int32_t level_start[MAXL + 1];
    DevDesc d[MAXD];
};

// ---------------------------------------------------------------------------
// Format constants
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int blk_bytes(int t) {
    return t == QDQ_Q4_K ? 144 : t == QDQ_Q6_K ? 210 : t == QDQ_Q8_0 ? 36 : 18;
}
__host__ __device__ constexpr int blk_weights(int t) { return (t == QDQ_Q4_K || t == QDQ_Q6_K) ? 256 : 32; }
__host__ __device__ constexpr int x_kind(int t) { return t == QDQ_Q4_K ? 1 : t == QDQ_Q4_0 ? 2 : 0; }

// ---------------------------------------------------------------------------
// Producer: bulk copies of a tile's bytes into a stage.
// Copies [floor16(src), min(ceil16(end), floor16(W_end))) in bulk and any last
// bytes of the matrix (past its final 16-byte boundary) with plain loads. The
// over-read bytes lie inside the matrix, so every access stays in bounds.
// mode kTail: store the trailing bytes (before the stage is released to the
// consumers by the arrive); mode kBulk: issue the bulk copy. Both return the
// bulk byte count.
// ---------------------------------------------------------------------------
constexpr int kTail = 1, kBulk = 2;

QDQ_DEV uint32_t copy_span(const uint8_t *src, uint32_t len, const uint8_t *w_end, uint32_t dst,
                           uint32_t bar, int mode) {
    const uintptr_t s = (uintptr_t)src, e = s + len;
    const uintptr_t a = s & ~(uintptr_t)15;
    const uintptr_t wend16 = (uintptr_t)w_end & ~(uintptr_t)15;
    uintptr_t b = (e + 15) & ~(uintptr_t)15;
    if (b > wend16) b = wend16 > a ? wend16 : a;
    if ((mode & kBulk) && b > a) bulk_g2s_hint(dst, (const void *)a, (uint32_t)(b - a), bar, policy_evict_first());
    if ((mode & kTail) && e > b) {  // at most 15 trailing bytes of the matrix
        for (uintptr_t p = b; p < e; ++p)
            asm volatile("st.shared.u8 [%0], %1;" ::"r"(dst + (uint32_t)(p - a)),
                         "h"((unsigned short)*(const uint8_t *)p)
                         : "memory");
    }
    return (uint32_t)(b - a);
}

// ---------------------------------------------------------------------------
// Consumer: per-format work on NR rows x the lane's 64 columns, batch 1.
//   wrow[r]: first byte of the unit's super-block (Q4_K, Q6_K) or block pair
//            (q8_0, q4_0) in row r, in shared memory.
//   xr:      the lane's 64 x values as 32 float pairs (pre-scaled for the nibble
//            formats) and, for Q4_K, the sums of x over its two sub-blocks;
//            shared by the NR rows.
// Shared memory is read with plain loads through pointers into the dynamic
// shared array, so the compiler can interleave the rows' loads and arithmetic.
// ---------------------------------------------------------------------------
struct XSlice {
    uint64_t v[32];
    float s0, s1;
};

QDQ_DEV uint4 ld4(const void *p) { return *(const uint4 *)p; }

// n consecutive 32-bit words at a 2-byte-aligned shared address: the covering
// 4-byte-aligned words, realigned with funnel shifts.
template <int N>
QDQ_DEV void ld_words_a2(const uint8_t *p, uint32_t (&out)[N]) {
    const uint32_t mis = (uint32_t)(uintptr_t)p & 3u;
    const uint32_t *base = (const uint32_t *)(p - mis);
    const uint32_t sh = mis * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = base[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// Q4_K: lane = 4 s + c covers chunk c of super-block s: sub-block 2c (low nibbles,
// x[0..31] of the slice) and 2c+1 (high nibbles, x[32..63]). Each sub-block is
// recentred (q4k_center): with s = d sc, m = dmin mn and rho its integer offset,
// sum = s_lo * sum((q - rho_lo) x)_lo + s_hi * sum((q - rho_hi) x)_hi
//       - (m_lo - s_lo rho_lo) * sum(x)_lo - (m_hi - s_hi rho_hi) * sum(x)_hi.
// A nibble left at bit position p reads as 2^23 + q 2^p; subtracting 2^23 + rho 2^p
// leaves (q - rho) 2^p exactly, against x pre-scaled by 2^-p.
template <int NR>
QDQ_DEV void unit_q4k(const uint8_t *const *wrow, int lane, const XSlice &xr, float (&out)[NR]) {
    const int s = lane >> 2, c = lane & 3;
    uint4 H[NR], Qa[NR], Qb[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const uint8_t *sb = wrow[r] + 144 * s;
        H[r] = ld4(sb);
        Qa[r] = ld4(sb + 16 + 32 * c);
        Qb[r] = ld4(sb + 32 + 32 * c);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        uint32_t sc2, mn2;
        q4k_pair_fields(H[r].y, H[r].z, H[r].w, c, &sc2, &mn2);
        const float d = half_bits_to_float(H[r].x & 0xFFFF), dmin = half_bits_to_float(H[r].x >> 16);
        const float s_lo = d * (float)(sc2 & 0xFF), s_hi = d * (float)(sc2 >> 8);
        float m_lo, m_hi;
        const float r_lo = q4k_center(s_lo, dmin * (float)(mn2 & 0xFF), &m_lo);
        const float r_hi = q4k_center(s_hi, dmin * (float)(mn2 >> 8), &m_hi);
        // 2^23 + rho 2^p for the nibble positions of each pair (0, 8), (16, 8), (4, 12)
        const uint64_t C_a = pack2(fmaf(r_lo, 1.0f, kTwo23), fmaf(r_lo, 256.0f, kTwo23));
        const uint64_t C_b = pack2(fmaf(r_lo, 65536.0f, kTwo23), fmaf(r_lo, 256.0f, kTwo23));
        const uint64_t C_h = pack2(fmaf(r_hi, 16.0f, kTwo23), fmaf(r_hi, 4096.0f, kTwo23));
        const uint32_t w[8] = {Qa[r].x, Qa[r].y, Qa[r].z, Qa[r].w, Qb[r].x, Qb[r].y, Qb[r].z, Qb[r].w};
        uint64_t a0 = 0, a1 = 0, h0 = 0, h1 = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t v = w[t], u = v >> 16;
            a0 = ffma2(fsub2(bits2(mask_magic<0xFu>(v), mask_magic<0xF00u>(v)), C_a), xr.v[2 * t], a0);
            a1 = ffma2(fsub2(bits2(mask_magic<0xF0000u>(v), mask_magic<0xF00u>(u)), C_b), xr.v[2 * t + 1], a1);
            h0 = ffma2(fsub2(bits2(mask_magic<0xF0u>(v), mask_magic<0xF000u>(v)), C_h), xr.v[16 + 2 * t], h0);
            h1 = ffma2(fsub2(bits2(mask_magic<0xF0u>(u), mask_magic<0xF000u>(u)), C_h), xr.v[17 + 2 * t], h1);
        }
        const float lo = (lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1));
        const float hi = (lo_of(h0) + hi_of(h0)) + (lo_of(h1) + hi_of(h1));
        out[r] = (s_lo * lo + s_hi * hi) - (m_lo * xr.s0 + m_hi * xr.s1);
    }
}

// Q6_K: lane = 4 s + 2 h + m covers, in super-block s, half h and the 16-wide
// column group m of each of the four 32-runs k: elements 128h + 32k + 16m + l,
// l < 16, with scale scales[8h + 2k + m] (= element / 16).
template <int NR>
QDQ_DEV void unit_q6k(const uint8_t *const *wrow, int lane, const XSlice &xr, float (&out)[NR]) {
    const int s = lane >> 2, h = (lane >> 1) & 1, m = lane & 1;
    uint32_t ql0[NR][4], ql1[NR][4], qh[NR][4], scw[NR][2], dw[NR][1];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const uint8_t *sb = wrow[r] + 210 * s;  // 2-byte aligned
        ld_words_a2<4>(sb + 64 * h + 16 * m, ql0[r]);
        ld_words_a2<4>(sb + 64 * h + 32 + 16 * m, ql1[r]);
        ld_words_a2<4>(sb + 128 + 32 * h + 16 * m, qh[r]);
        ld_words_a2<2>(sb + 192 + 8 * h, scw[r]);
        ld_words_a2<1>(sb + 208, dw[r]);
    }
    const uint64_t M32 = bits2(__float_as_uint(kTwo23 + 32.0f), __float_as_uint(kTwo23 + 32.0f));
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float d = half_bits_to_float(dw[r][0] & 0xFFFF);
        float sc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int byte = m + 2 * k;  // byte index within scw
            const uint32_t word = byte < 4 ? scw[r][0] : scw[r][1];
            sc[k] = (float)(int)(int8_t)((word >> (8 * (byte & 3))) & 0xFF);
        }
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint64_t a0 = 0, a1 = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t b6 = q6k_quant_bytes((k & 1) ? ql1[r][t] : ql0[r][t], qh[r][t], k);
                a0 = ffma2(fsub2(bits2(byte_to_magic<0>(b6), byte_to_magic<1>(b6)), M32), xr.v[8 * k + 2 * t], a0);
                a1 = ffma2(fsub2(bits2(byte_to_magic<2>(b6), byte_to_magic<3>(b6)), M32), xr.v[8 * k + 2 * t + 1], a1);
            }
            sum += sc[k] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
        }
        out[r] = d * sum;
    }
}

// q8_0: lane covers blocks 2*lane and 2*lane+1 of the slice (x[0..31], x[32..63]
// of its 64). An int8 q becomes 2^23 + (q + 128) by flipping its sign bit and
// placing the byte under the exponent; subtracting 2^23 + 128 leaves q exactly.
template <int NR>
QDQ_DEV void unit_q8_0(const uint8_t *const *wrow, int lane, int nblk_valid, const XSlice &xr, float (&out)[NR]) {
    const uint64_t M128 = bits2(__float_as_uint(kTwo23 + 128.0f), __float_as_uint(kTwo23 + 128.0f));
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        float d[2];
        uint64_t q[32];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t *base = (const uint32_t *)(wrow[r] + 72 * lane + 36 * i);  // 4-byte aligned
            const bool valid = 2 * lane + i < nblk_valid;
            d[i] = valid ? __uint_as_float(base[0]) : 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t v = valid ? (base[1 + t] ^ 0x80808080u) : 0x80808080u;
                q[16 * i + 2 * t] = fsub2(bits2(byte_to_magic<0>(v), byte_to_magic<1>(v)), M128);
                q[16 * i + 2 * t + 1] = fsub2(bits2(byte_to_magic<2>(v), byte_to_magic<3>(v)), M128);
            }
        }
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint64_t a0 = 0, a1 = 0;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                a0 = ffma2(q[16 * i + j], xr.v[16 * i + j], a0);
                a1 = ffma2(q[16 * i + j + 1], xr.v[16 * i + j + 1], a1);
            }
            sum += d[i] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
        }
        out[r] = sum;
    }
}

// q4_0: lane covers blocks 2*lane, 2*lane+1 (36 bytes, 2-byte aligned). Byte i
// of a block holds weight i (low nibble) and weight i+16 (high nibble). Nibbles
// stay at their bit position p (x pre-scaled by 2^-p); subtracting 2^23 + 8*2^p
// gives (q - 8) * 2^p exactly.
template <int NR>
QDQ_DEV void unit_q4_0(const uint8_t *const *wrow, int lane, int nblk_valid, const XSlice &xr, float (&out)[NR]) {
    const uint64_t C_la = bits2(__float_as_uint(kTwo23 + 8.0f), __float_as_uint(kTwo23 + 2048.0f));
    const uint64_t C_lb = bits2(__float_as_uint(kTwo23 + 524288.0f), __float_as_uint(kTwo23 + 2048.0f));
    const uint64_t C_h = bits2(__float_as_uint(kTwo23 + 128.0f), __float_as_uint(kTwo23 + 32768.0f));
    const bool v0 = 2 * lane < nblk_valid, v1 = 2 * lane + 1 < nblk_valid;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        uint32_t w[9];
        if (v1) {
            ld_words_a2<9>(wrow[r] + 36 * lane, w);
        } else {  // only the first block is inside the row segment
            uint32_t w5[5];
            ld_words_a2<5>(wrow[r] + 36 * lane, w5);
#pragma unroll
            for (int i = 0; i < 5; ++i) w[i] = w5[i];
#pragma unroll
            for (int i = 5; i < 9; ++i) w[i] = 0x88888888u;
        }
        float d[2];
        d[0] = v0 ? half_bits_to_float(w[0] & 0xFFFF) : 0.f;
        d[1] = v1 ? half_bits_to_float(w[4] >> 16) : 0.f;
        uint32_t qs[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) qs[t] = __funnelshift_r(w[t], w[t + 1], 16);
#pragma unroll
        for (int t = 0; t < 4; ++t) qs[4 + t] = w[5 + t];
        uint64_t q[32];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t v = qs[4 * i + t], u = v >> 16;
                q[16 * i + 2 * t] = fsub2(bits2(mask_magic<0xFu>(v), mask_magic<0xF00u>(v)), C_la);
                q[16 * i + 2 * t + 1] = fsub2(bits2(mask_magic<0xF0000u>(v), mask_magic<0xF00u>(u)), C_lb);
                q[16 * i + 8 + 2 * t] = fsub2(bits2(mask_magic<0xF0u>(v), mask_magic<0xF000u>(v)), C_h);
                q[16 * i + 9 + 2 * t] = fsub2(bits2(mask_magic<0xF0u>(u), mask_magic<0xF000u>(u)), C_h);
            }
        }
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint64_t a0 = 0, a1 = 0;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                a0 = ffma2(q[16 * i + j], xr.v[16 * i + j], a0);
                a1 = ffma2(q[16 * i + j + 1], xr.v[16 * i + j + 1], a1);
            }
            sum += d[i] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
        }
        out[r] = sum;
    }
}

// Scale that puts x next to a nibble read at its bit position (see unit_q4k /
// unit_q4_0): low nibbles of bytes 0..3 of a word sit at bits 0, 8, 16, 8 (the
// last after a 16-bit shift), high nibbles at bits 4, 12, 4, 12.
QDQ_DEV float nibble_scale(bool high, int p) {
    const float lo = p == 0 ? 1.f : p == 2 ? 1.52587890625e-05f : 0.00390625f;
    const float hi = (p & 1) ? 0.000244140625f : 0.0625f;
    return high ? hi : lo;
}

}  // namespace qdq
