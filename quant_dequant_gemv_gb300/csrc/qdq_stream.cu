// qdq_stream.cu -- fused dequant-GEMV on CUDA cores, batch 1..8.
//
// "S21 The Capstone: picoLM, in Python", section 3 (fused dequant + dot: walk
// the quantised bytes and accumulate the dot product while decoding, so only
// the 4-bit data crosses the memory bus) and section 4 (model_forward: the
// per-layer projections of a decode step); "PETIT" (gemv_q8 / gemv_q4, weights
// stored out x in).
//
// Design (one persistent CTA per SM, warp-specialised):
//  * Work: a list of GEMVs in dependency levels. In each level the level's rows
//    are split across CTAs by weight bytes; each CTA walks its rows in tiles of
//    whole rows (or row segments, when a column chunk is needed) that fit one
//    32 KiB shared-memory stage.
//  * Warp 0 (producer) streams tile bytes HBM -> shared memory with 1-D bulk
//    copies (cp.async.bulk, no multicast) into a ring of stages guarded by
//    full/empty mbarriers. It never waits for level dependencies: weights do
//    not depend on earlier outputs, so it runs ahead into later levels.
//  * Warps 1..8 (consumers) wait for the level's input to be ready (a counter
//    per level, bounded wait), stage x (and the Q4_K sub-block sums of x) in
//    shared memory, then decode and multiply. A lane covers 64 weights of a
//    2048-column block of one row; for batch 1 its 64 x values stay in
//    registers across rows. Nibbles and 6-bit quants become floats by
//    exponent-field construction (no int->float conversions per weight), and
//    the products accumulate with packed f32x2 FMAs. Per-row sums go through a
//    warp shuffle tree and a fixed-order cross-warp sum, so results are
//    deterministic.
//  * Every wait is bounded (qdq_device.cuh).
#include <cstdio>
#include <cstring>
#include <new>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {

static __device__ int s_status_stream;

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;
constexpr int kStageBytes = 32768;
constexpr int kCB = 2048;      // columns per column block (32 lanes x 64)
constexpr int kUnitsMax = 256;  // (row, column block) units per tile
constexpr int kXSumFloats = 512;

template <int BT> struct Cfg;
template <> struct Cfg<1> { static constexpr int kStages = 5; static constexpr int kXBytes = 57344; };
template <> struct Cfg<2> { static constexpr int kStages = 4; static constexpr int kXBytes = 65536; };
template <> struct Cfg<4> { static constexpr int kStages = 4; static constexpr int kXBytes = 65536; };
template <> struct Cfg<8> { static constexpr int kStages = 4; static constexpr int kXBytes = 65536; };

template <int BT>
constexpr int smem_bytes() {
    return Cfg<BT>::kStages * kStageBytes + Cfg<BT>::kXBytes + kXSumFloats * 4 + 2 * kUnitsMax * BT * 4 +
           2 * Cfg<BT>::kStages * 8;
}

struct DevDesc {
    const uint8_t *W;
    const float *x;
    float *y;
    int64_t rows;
    int32_t cols;
    int32_t type;
    int32_t rb;     // bytes per row
    int32_t kc;     // columns per chunk
    int32_t kinds;  // bit k set: this x needs staged copy kind k (0 plain, 1 Q4_K-scaled, 2 q4_0-scaled)
    int32_t pad;
};

template <int MAXD, int MAXL>
struct StreamArgs {
    int32_t ndesc, nlevels, batch, pad;
    unsigned *counters;
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
// Tile walk: identical sequence for the producer and the consumers.
// ---------------------------------------------------------------------------
struct Tile {
    int g;
    int nrows;
    int64_t row0;
    int kc0, kcols;
    bool contiguous;
};

struct TileGeom {
    int ncb;       // column blocks in this chunk
    int segbytes;  // bytes of one row segment
    int pitch;     // slot pitch in chunk mode
    int rmax;      // rows per tile
};

QDQ_DEV TileGeom tile_geom(const DevDesc &d, int kcols, bool contiguous) {
    TileGeom t;
    t.ncb = (kcols + kCB - 1) / kCB;
    t.segbytes = (kcols / blk_weights(d.type)) * blk_bytes(d.type);
    t.pitch = ((t.segbytes + 15) & ~15) + 16;
    int r_units = kUnitsMax / t.ncb;
    int r_bytes = contiguous ? (kStageBytes - 32) / d.rb : kStageBytes / t.pitch;
    t.rmax = r_units < r_bytes ? r_units : r_bytes;
    if (t.rmax < 1) t.rmax = 1;
    return t;
}

// Rows [ra, rb) of desc g that this CTA owns in its level (byte-balanced split).
template <class A>
QDQ_DEV void cta_rows(const A &a, int L, int g, int cta, int P, int64_t *ra, int64_t *rb) {
    int64_t total = 0, start = 0;
    for (int i = a.level_start[L]; i < a.level_start[L + 1]; ++i) {
        const int64_t bytes = a.d[i].rows * (int64_t)a.d[i].rb;
        if (i < g) start += bytes;
        total += bytes;
    }
    const int64_t A0 = (int64_t)cta * total / P, B0 = (int64_t)(cta + 1) * total / P;
    const int64_t rbytes = a.d[g].rb, rows = a.d[g].rows;
    auto row_at = [&](int64_t byte) -> int64_t {
        int64_t off = byte - start;
        if (off <= 0) return 0;
        int64_t r = (off + rbytes - 1) / rbytes;
        return r < rows ? r : rows;
    };
    *ra = row_at(A0);
    *rb = row_at(B0);
}

template <class A, class FBegin, class FTile, class FEnd>
QDQ_DEV void walk(const A &a, int cta, int P, FBegin &&on_begin, FTile &&on_tile, FEnd &&on_end) {
    for (int L = 0; L < a.nlevels; ++L) {
        on_begin(L);
        for (int g = a.level_start[L]; g < a.level_start[L + 1]; ++g) {
            const DevDesc &d = a.d[g];
            int64_t ra, rb;
            cta_rows(a, L, g, cta, P, &ra, &rb);
            if (ra >= rb) continue;
            for (int kc0 = 0; kc0 < d.cols; kc0 += d.kc) {
                const int kcols = d.cols - kc0 < d.kc ? d.cols - kc0 : d.kc;
                const bool contiguous = (kc0 == 0 && kcols == d.cols);
                const TileGeom geo = tile_geom(d, kcols, contiguous);
                for (int64_t r0 = ra; r0 < rb; r0 += geo.rmax) {
                    Tile t;
                    t.g = g;
                    t.row0 = r0;
                    t.nrows = (int)(rb - r0 < geo.rmax ? rb - r0 : geo.rmax);
                    t.kc0 = kc0;
                    t.kcols = kcols;
                    t.contiguous = contiguous;
                    on_tile(t, geo);
                }
            }
        }
        on_end(L);
    }
}

// ---------------------------------------------------------------------------
// Producer: bulk copies of a tile's bytes into a stage.
// Copies [floor16(src), min(ceil16(end), floor16(W_end))) in bulk and any last
// bytes of the matrix (past its final 16-byte boundary) with plain loads. The
// over-read bytes lie inside the matrix, so every access stays in bounds.
// ---------------------------------------------------------------------------
// mode kTail: store the trailing bytes (before the stage is released to the
// consumers by the arrive); mode kBulk: issue the bulk copy. Both return the
// bulk byte count.
constexpr int kTail = 1, kBulk = 2;

QDQ_DEV uint32_t copy_span(const uint8_t *src, uint32_t len, const uint8_t *w_end, uint32_t dst,
                           uint32_t bar, int mode) {
    const uintptr_t s = (uintptr_t)src, e = s + len;
    const uintptr_t a = s & ~(uintptr_t)15;
    const uintptr_t wend16 = (uintptr_t)w_end & ~(uintptr_t)15;
    uintptr_t b = (e + 15) & ~(uintptr_t)15;
    if (b > wend16) b = wend16 > a ? wend16 : a;
    if ((mode & kBulk) && b > a) bulk_g2s(dst, (const void *)a, (uint32_t)(b - a), bar);
    if ((mode & kTail) && e > b) {  // at most 15 trailing bytes of the matrix
        for (uintptr_t p = b; p < e; ++p)
            asm volatile("st.shared.u8 [%0], %1;" ::"r"(dst + (uint32_t)(p - a)),
                         "h"((unsigned short)*(const uint8_t *)p)
                         : "memory");
    }
    return (uint32_t)(b - a);
}

QDQ_DEV uint32_t tile_bytes(const DevDesc &d, const Tile &t, const TileGeom &geo, uint32_t stage, uint32_t bar,
                            int mode) {
    const uint8_t *w_end = d.W + d.rows * (int64_t)d.rb;
    if (t.contiguous) {
        return copy_span(d.W + t.row0 * d.rb, (uint32_t)t.nrows * d.rb, w_end, stage, bar, mode);
    }
    uint32_t total = 0;
    const int64_t off = (int64_t)(t.kc0 / blk_weights(d.type)) * blk_bytes(d.type);
    for (int r = 0; r < t.nrows; ++r)
        total += copy_span(d.W + (t.row0 + r) * d.rb + off, (uint32_t)geo.segbytes, w_end,
                           stage + (uint32_t)(r * geo.pitch), bar, mode);
    return total;
}

// ---------------------------------------------------------------------------
// Consumer: per-format work on one (row, column block) unit.
//   wrow: shared address of the first byte of this column block in the row.
//   xs:   shared address of this lane's x slice in the matching staged copy
//         (batch 0); batch b is at xs + b * xstride.
//   xr:   batch 1 only: the lane's 64 x values as 32 float pairs.
// ---------------------------------------------------------------------------
struct XSlice {
    uint64_t v[32];
    float s0, s1;  // Q4_K: sums of x over the lane's two sub-blocks
};

QDQ_DEV void load_pairs16(uint32_t a, uint64_t *dst) {  // 16 floats -> 8 pairs
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = lds128(a + 16 * i);
        dst[2 * i] = bits2(v.x, v.y);
        dst[2 * i + 1] = bits2(v.z, v.w);
    }
}

// x slice offsets (in floats, relative to the column block start) per format.
template <int TYPE>
QDQ_DEV int lane_col0(int lane) {
    if constexpr (TYPE == QDQ_Q4_K) return 256 * (lane >> 2) + 64 * (lane & 3);
    else if constexpr (TYPE == QDQ_Q6_K) return 256 * (lane >> 2) + 128 * ((lane >> 1) & 1) + 16 * (lane & 1);
    else return 64 * lane;
}

template <int TYPE>
QDQ_DEV void load_x(uint32_t xs, uint32_t xsum_addr, XSlice &x) {
    if constexpr (TYPE == QDQ_Q6_K) {  // four runs of 16 at stride 32
#pragma unroll
        for (int k = 0; k < 4; ++k) load_pairs16(xs + 128 * k, &x.v[8 * k]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) load_pairs16(xs + 64 * k, &x.v[8 * k]);
    }
    if constexpr (TYPE == QDQ_Q4_K) {
        x.s0 = ldsf(xsum_addr);
        x.s1 = ldsf(xsum_addr + 4);
    }
}

template <int BT>
struct Acc {
    float v[BT];
};

// Q4_K: lane = 4 s + c covers chunk c of super-block s: sub-block 2c (low nibbles,
// x[0..31] of the slice) and 2c+1 (high nibbles, x[32..63]).
// sum = d * (sc_lo * sum(q x)_lo + sc_hi * sum(q x)_hi) - dmin * (mn_lo * sum(x)_lo + mn_hi * sum(x)_hi)
template <int BT>
QDQ_DEV void unit_q4k(uint32_t wrow, int lane, const XSlice &xr, uint32_t xs, uint32_t xstride,
                      uint32_t xsum_addr, uint32_t xsum_stride, Acc<BT> &out) {
    const int s = lane >> 2, c = lane & 3;
    const uint32_t sb = wrow + 144 * s;
    const uint4 H = lds128(sb);
    const uint4 Qa = lds128(sb + 16 + 32 * c), Qb = lds128(sb + 32 + 32 * c);
    uint32_t sc2, mn2;
    q4k_pair_fields(H.y, H.z, H.w, c, &sc2, &mn2);
    const float d = half_bits_to_float(H.x & 0xFFFF), dmin = half_bits_to_float(H.x >> 16);
    const float sc_lo = (float)(sc2 & 0xFF), sc_hi = (float)(sc2 >> 8);
    const float mn_lo = (float)(mn2 & 0xFF), mn_hi = (float)(mn2 >> 8);
    const uint32_t w[8] = {Qa.x, Qa.y, Qa.z, Qa.w, Qb.x, Qb.y, Qb.z, Qb.w};
    const uint64_t M2 = bits2(__float_as_uint(kTwo23), __float_as_uint(kTwo23));
    uint64_t q[32];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t v = w[t], u = v >> 16;
        q[2 * t] = fsub2(bits2((v & 0xFu) | kMagic, (v & 0xF00u) | kMagic), M2);
        q[2 * t + 1] = fsub2(bits2((v & 0xF0000u) | kMagic, (u & 0xF00u) | kMagic), M2);
        q[16 + 2 * t] = fsub2(bits2((v & 0xF0u) | kMagic, (v & 0xF000u) | kMagic), M2);
        q[17 + 2 * t] = fsub2(bits2((u & 0xF0u) | kMagic, (u & 0xF000u) | kMagic), M2);
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        uint64_t a0 = 0, a1 = 0, h0 = 0, h1 = 0;
        if constexpr (BT == 1) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                a0 = ffma2(q[i], xr.v[i], a0);
                a1 = ffma2(q[i + 1], xr.v[i + 1], a1);
                h0 = ffma2(q[16 + i], xr.v[16 + i], h0);
                h1 = ffma2(q[17 + i], xr.v[17 + i], h1);
            }
            const float lo = (lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1));
            const float hi = (lo_of(h0) + hi_of(h0)) + (lo_of(h1) + hi_of(h1));
            out.v[b] = d * (sc_lo * lo + sc_hi * hi) - dmin * (mn_lo * xr.s0 + mn_hi * xr.s1);
        } else {
            const uint32_t xb = xs + b * xstride;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const uint4 xl0 = lds128(xb + 8 * i), xl1 = lds128(xb + 8 * i + 16);
                const uint4 xh0 = lds128(xb + 128 + 8 * i), xh1 = lds128(xb + 128 + 8 * i + 16);
                a0 = ffma2(q[i], bits2(xl0.x, xl0.y), a0);
                a1 = ffma2(q[i + 1], bits2(xl0.z, xl0.w), a1);
                a0 = ffma2(q[i + 2], bits2(xl1.x, xl1.y), a0);
                a1 = ffma2(q[i + 3], bits2(xl1.z, xl1.w), a1);
                h0 = ffma2(q[16 + i], bits2(xh0.x, xh0.y), h0);
                h1 = ffma2(q[17 + i], bits2(xh0.z, xh0.w), h1);
                h0 = ffma2(q[18 + i], bits2(xh1.x, xh1.y), h0);
                h1 = ffma2(q[19 + i], bits2(xh1.z, xh1.w), h1);
            }
            const float lo = (lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1));
            const float hi = (lo_of(h0) + hi_of(h0)) + (lo_of(h1) + hi_of(h1));
            const float s0 = ldsf(xsum_addr + b * xsum_stride), s1 = ldsf(xsum_addr + b * xsum_stride + 4);
            out.v[b] = d * (sc_lo * lo + sc_hi * hi) - dmin * (mn_lo * s0 + mn_hi * s1);
        }
    }
}

// Q6_K: lane = 4 s + 2 h + m covers, in super-block s, half h and the 16-wide
// column group m of each of the four 32-runs k: elements 128h + 32k + 16m + l,
// l < 16, with scale scales[8h + 2k + m] (= element / 16).
template <int BT>
QDQ_DEV void unit_q6k(uint32_t wrow, int lane, const XSlice &xr, uint32_t xs, uint32_t xstride,
                      Acc<BT> &out) {
    const int s = lane >> 2, h = (lane >> 1) & 1, m = lane & 1;
    const uint32_t sb = wrow + 210 * s;  // 2-byte aligned
    uint32_t ql0[4], ql1[4], qh[4], scw[2], dw[1];
    lds_words_a2<4>(sb + 64 * h + 16 * m, ql0);
    lds_words_a2<4>(sb + 64 * h + 32 + 16 * m, ql1);
    lds_words_a2<4>(sb + 128 + 32 * h + 16 * m, qh);
    lds_words_a2<2>(sb + 192 + 8 * h, scw);
    lds_words_a2<1>(sb + 208, dw);
    const float d = half_bits_to_float(dw[0] & 0xFFFF);
    float sc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int byte = m + 2 * k;  // byte index within scw
        const uint32_t word = byte < 4 ? scw[0] : scw[1];
        sc[k] = (float)(int)(int8_t)((word >> (8 * (byte & 3))) & 0xFF);
    }
    const uint64_t M32 = bits2(__float_as_uint(kTwo23 + 32.0f), __float_as_uint(kTwo23 + 32.0f));
    uint64_t q[32];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t b6 = q6k_quant_bytes((k & 1) ? ql1[t] : ql0[t], qh[t], k);
            q[8 * k + 2 * t] = fsub2(bits2(byte_to_magic<0>(b6), byte_to_magic<1>(b6)), M32);
            q[8 * k + 2 * t + 1] = fsub2(bits2(byte_to_magic<2>(b6), byte_to_magic<3>(b6)), M32);
        }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint64_t a0 = 0, a1 = 0;
            if constexpr (BT == 1) {
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    a0 = ffma2(q[8 * k + i], xr.v[8 * k + i], a0);
                    a1 = ffma2(q[8 * k + i + 1], xr.v[8 * k + i + 1], a1);
                }
            } else {
                const uint32_t xb = xs + b * xstride + 128 * k;
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const uint4 xv = lds128(xb + 8 * i);
                    a0 = ffma2(q[8 * k + i], bits2(xv.x, xv.y), a0);
                    a1 = ffma2(q[8 * k + i + 1], bits2(xv.z, xv.w), a1);
                }
            }
            sum += sc[k] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
        }
        out.v[b] = d * sum;
    }
}

// q8_0: lane covers blocks 2*lane and 2*lane+1 of the column block (x[0..31],
// x[32..63] of the slice). An int8 q becomes 2^23 + (q + 128) by flipping its
// sign bit and placing the byte under the exponent; subtracting 2^23 + 128
// leaves q exactly.
template <int BT>
QDQ_DEV void unit_q8_0(uint32_t wrow, int lane, int nblk_valid, const XSlice &xr, uint32_t xs,
                       uint32_t xstride, Acc<BT> &out) {
    const uint64_t M128 = bits2(__float_as_uint(kTwo23 + 128.0f), __float_as_uint(kTwo23 + 128.0f));
    float d[2];
    uint64_t q[32];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t base = wrow + 72 * lane + 36 * i;  // 4-byte aligned
        const bool valid = 2 * lane + i < nblk_valid;
        d[i] = valid ? __uint_as_float(lds32(base)) : 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t v = valid ? (lds32(base + 4 + 4 * t) ^ 0x80808080u) : 0x80808080u;
            q[16 * i + 2 * t] = fsub2(bits2(byte_to_magic<0>(v), byte_to_magic<1>(v)), M128);
            q[16 * i + 2 * t + 1] = fsub2(bits2(byte_to_magic<2>(v), byte_to_magic<3>(v)), M128);
        }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint64_t a0 = 0, a1 = 0;
            if constexpr (BT == 1) {
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    a0 = ffma2(q[16 * i + j], xr.v[16 * i + j], a0);
                    a1 = ffma2(q[16 * i + j + 1], xr.v[16 * i + j + 1], a1);
                }
            } else {
                const uint32_t xb = xs + b * xstride + 128 * i;
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const uint4 xv = lds128(xb + 8 * j);
                    a0 = ffma2(q[16 * i + j], bits2(xv.x, xv.y), a0);
                    a1 = ffma2(q[16 * i + j + 1], bits2(xv.z, xv.w), a1);
                }
            }
            sum += d[i] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
        }
        out.v[b] = sum;
    }
}

// q4_0: lane covers blocks 2*lane, 2*lane+1 (36 bytes, 2-byte aligned). Byte i
// of a block holds weight i (low nibble) and weight i+16 (high nibble). Nibbles
// stay at their bit position p (x pre-scaled by 2^-p); subtracting 2^23 + 8*2^p
// gives (q - 8) * 2^p exactly.
template <int BT>
QDQ_DEV void unit_q4_0(uint32_t wrow, int lane, int nblk_valid, const XSlice &xr, uint32_t xs,
                       uint32_t xstride, Acc<BT> &out) {
    const uint64_t C_la = bits2(__float_as_uint(kTwo23 + 8.0f), __float_as_uint(kTwo23 + 2048.0f));
    const uint64_t C_lb = bits2(__float_as_uint(kTwo23 + 524288.0f), __float_as_uint(kTwo23 + 2048.0f));
    const uint64_t C_h = bits2(__float_as_uint(kTwo23 + 128.0f), __float_as_uint(kTwo23 + 32768.0f));
    float d[2];
    uint64_t q[32];
    uint32_t w[9];
    const bool v0 = 2 * lane < nblk_valid, v1 = 2 * lane + 1 < nblk_valid;
    if (v1) {
        lds_words_a2<9>(wrow + 36 * lane, w);
    } else if (v0) {  // only the first block is inside the row segment
        uint32_t w5[5];
        lds_words_a2<5>(wrow + 36 * lane, w5);
#pragma unroll
        for (int i = 0; i < 5; ++i) w[i] = w5[i];
#pragma unroll
        for (int i = 5; i < 9; ++i) w[i] = 0x88888888u;
    } else {
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = 0x88888888u;
    }
    d[0] = v0 ? half_bits_to_float(w[0] & 0xFFFF) : 0.f;
    d[1] = v1 ? half_bits_to_float(w[4] >> 16) : 0.f;
    uint32_t qs[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) qs[t] = __funnelshift_r(w[t], w[t + 1], 16);
#pragma unroll
    for (int t = 0; t < 4; ++t) qs[4 + t] = w[5 + t];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t v = qs[4 * i + t], u = v >> 16;
            q[16 * i + 2 * t] = fsub2(bits2((v & 0xFu) | kMagic, (v & 0xF00u) | kMagic), C_la);
            q[16 * i + 2 * t + 1] = fsub2(bits2((v & 0xF0000u) | kMagic, (u & 0xF00u) | kMagic), C_lb);
            q[16 * i + 8 + 2 * t] = fsub2(bits2((v & 0xF0u) | kMagic, (v & 0xF000u) | kMagic), C_h);
            q[16 * i + 9 + 2 * t] = fsub2(bits2((u & 0xF0u) | kMagic, (u & 0xF000u) | kMagic), C_h);
        }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint64_t a0 = 0, a1 = 0;
            if constexpr (BT == 1) {
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    a0 = ffma2(q[16 * i + j], xr.v[16 * i + j], a0);
                    a1 = ffma2(q[16 * i + j + 1], xr.v[16 * i + j + 1], a1);
                }
            } else {
                const uint32_t xb = xs + b * xstride + 128 * i;
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const uint4 xv = lds128(xb + 8 * j);
                    a0 = ffma2(q[16 * i + j], bits2(xv.x, xv.y), a0);
                    a1 = ffma2(q[16 * i + j + 1], bits2(xv.z, xv.w), a1);
                }
            }
            sum += d[i] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
        }
        out.v[b] = sum;
    }
}

QDQ_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Scale that puts x next to a nibble read at its bit position (see unit_q4k /
// unit_q4_0): low nibbles of bytes 0..3 of a word sit at bits 0, 8, 16, 8 (the
// last after a 16-bit shift), high nibbles at bits 4, 12, 4, 12.
QDQ_DEV float nibble_scale(bool high, int p) {
    const float lo[4] = {1.f, 0.00390625f, 1.52587890625e-05f, 0.00390625f};
    const float hi[4] = {0.0625f, 0.000244140625f, 0.0625f, 0.000244140625f};
    return high ? hi[p] : lo[p];
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int BT, int MAXD, int MAXL>
__global__ void __launch_bounds__(kThreads, 1)
    stream_kernel(const __grid_constant__ StreamArgs<MAXD, MAXL> a) {
    constexpr int NST = Cfg<BT>::kStages;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *ring = smem;
    float *xbuf = (float *)(smem + NST * kStageBytes);
    float *xsum = (float *)(smem + NST * kStageBytes + Cfg<BT>::kXBytes);
    float *partial = xsum + kXSumFloats;
    uint64_t *bars = (uint64_t *)(partial + 2 * kUnitsMax * BT);
    const uint32_t ring_a = smem_u32(ring), xbuf_a = smem_u32(xbuf), xsum_a = smem_u32(xsum);
    const uint32_t full_a = smem_u32(bars), empty_a = full_a + 8 * NST;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, P = gridDim.x;
    int *status = &s_status_stream;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full_a + 8 * s, 1);
            mbar_init(empty_a + 8 * s, 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        int t = 0;
        walk(
            a, cta, P, [](int) {},
            [&](const Tile &tl, const TileGeom &geo) {
                const int s = t % NST;
                if (t >= NST) mbar_wait(empty_a + 8 * s, ((t / NST) + 1) & 1, status);
                const DevDesc &d = a.d[tl.g];
                const uint32_t stage = ring_a + s * kStageBytes, bar = full_a + 8 * s;
                const uint32_t bytes = tile_bytes(d, tl, geo, stage, bar, kTail);
                mbar_arrive_expect_tx(bar, bytes);  // releases the tail stores above
                tile_bytes(d, tl, geo, stage, bar, kBulk);
                ++t;
            },
            [](int) {});
        // Do not leave while copies are in flight.
        for (int i = t - NST > 0 ? t - NST : 0; i < t; ++i)
            mbar_wait(full_a + 8 * (i % NST), (i / NST) & 1, status);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1, ctid = threadIdx.x - 32;
    int t = 0, pb = 0;
    // x staging state
    const float *st_x = nullptr;
    int st_kc0 = -1, st_epoch = 0;
    int kind_off[3] = {-1, -1, -1};  // float offset of each staged copy in xbuf
    int st_kc = 0;                   // columns per batch row of the staged chunk
    // lane x cache (batch 1)
    XSlice xr;
    int xr_epoch = -1, xr_j = -1, xr_type = -1;

    auto stage_x = [&](const DevDesc &d, int kc0, int kcols) {
        // All consumers have passed the barrier that ended the previous tile, so
        // nobody still reads the old x.
        int nk = 0;
        for (int k = 0; k < 3; ++k) kind_off[k] = (d.kinds >> k) & 1 ? (nk++) * kcols * BT : -1;
        st_kc = kcols;
        const int n4 = kcols / 4;
        for (int i = ctid; i < n4 * BT; i += kConsumers) {
            const int b = i / n4, k4 = i - b * n4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (b < a.batch) v = __ldcg((const float4 *)(d.x + (int64_t)b * d.cols + kc0) + k4);
            const int col = 4 * k4;
            if (kind_off[0] >= 0) *(float4 *)(xbuf + kind_off[0] + b * kcols + col) = v;
            if (kind_off[1] >= 0) {  // Q4_K: low nibbles are columns 0..31 of each 64
                const bool hi = (col & 63) >= 32;
                float4 w = make_float4(v.x * nibble_scale(hi, 0), v.y * nibble_scale(hi, 1),
                                       v.z * nibble_scale(hi, 2), v.w * nibble_scale(hi, 3));
                *(float4 *)(xbuf + kind_off[1] + b * kcols + col) = w;
            }
            if (kind_off[2] >= 0) {  // q4_0: low nibbles are columns 0..15 of each 32
                const bool hi = (col & 31) >= 16;
                float4 w = make_float4(v.x * nibble_scale(hi, 0), v.y * nibble_scale(hi, 1),
                                       v.z * nibble_scale(hi, 2), v.w * nibble_scale(hi, 3));
                *(float4 *)(xbuf + kind_off[2] + b * kcols + col) = w;
            }
        }
        if (kind_off[1] >= 0) {  // sums of x over each 32-column sub-block
            const int nsub = kcols / 32;
            for (int i = ctid; i < nsub * BT; i += kConsumers) {
                const int b = i / nsub, j = i - b * nsub;
                const float *src = d.x + (int64_t)b * d.cols + kc0 + 32 * j;
                float s = 0.f;
                if (b < a.batch) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 v = __ldcg((const float4 *)src + k);
                        s += (v.x + v.y) + (v.z + v.w);
                    }
                }
                xsum[b * nsub + j] = s;
            }
        }
        named_bar_sync(1, kConsumers);
        st_x = d.x;
        st_kc0 = kc0;
        ++st_epoch;
    };

    walk(
        a, cta, P,
        [&](int L) {
            if (L > 0 && a.counters != nullptr) {
                if (ctid == 0) wait_counter(&a.counters[L - 1], (unsigned)P, status, kWaitLimitNs);
                named_bar_sync(1, kConsumers);
            }
            st_x = nullptr;  // a new level's input must be staged after its dependency
        },
        [&](const Tile &tl, const TileGeom &geo) {
            const DevDesc &d = a.d[tl.g];
            if (d.x != st_x || tl.kc0 != st_kc0) stage_x(d, tl.kc0, tl.kcols);
            const int s = t % NST;
            mbar_wait(full_a + 8 * s, (t / NST) & 1, status);
            const uint32_t stage = ring_a + s * kStageBytes;
            const int nU = tl.nrows * geo.ncb;
            const int qk = blk_weights(d.type), bb = blk_bytes(d.type);
            const uint32_t cb_bytes = (uint32_t)(kCB / qk) * bb;
            float *pbuf = partial + pb * kUnitsMax * BT;
            for (int u = cw; u < nU; u += kConsumerWarps) {
                const int j = u / tl.nrows, r = u - j * tl.nrows;
                uint32_t wrow;
                if (tl.contiguous) {
                    const uint32_t delta = (uint32_t)((uintptr_t)(d.W + tl.row0 * d.rb) & 15);
                    wrow = stage + delta + (uint32_t)r * d.rb;
                } else {
                    const int64_t off = (int64_t)(tl.kc0 / qk) * bb;
                    const uint32_t delta = (uint32_t)((uintptr_t)(d.W + (tl.row0 + r) * d.rb + off) & 15);
                    wrow = stage + (uint32_t)r * geo.pitch + delta;
                }
                wrow += (uint32_t)j * cb_bytes;
                const int cols_here = tl.kcols - j * kCB < kCB ? tl.kcols - j * kCB : kCB;
                Acc<BT> acc;
                const int kind = x_kind(d.type);
                const uint32_t xstride = (uint32_t)st_kc * 4;
                const int xcol = j * kCB;
                if (d.type == QDQ_Q4_K) {
                    const int c0 = lane_col0<QDQ_Q4_K>(lane);
                    const uint32_t xs = xbuf_a + 4 * (kind_off[kind] + xcol + c0);
                    const uint32_t xsa = xsum_a + 4 * ((xcol + c0) / 32);
                    const uint32_t xss = (uint32_t)(st_kc / 32) * 4;
                    if (256 * (lane >> 2) < cols_here) {
                        if (BT == 1 && (xr_epoch != st_epoch || xr_j != j || xr_type != d.type)) {
                            load_x<QDQ_Q4_K>(xs, xsa, xr);
                            xr_epoch = st_epoch; xr_j = j; xr_type = d.type;
                        }
                        unit_q4k<BT>(wrow, lane, xr, xs, xstride, xsa, xss, acc);
                    } else {
#pragma unroll
                        for (int b = 0; b < BT; ++b) acc.v[b] = 0.f;
                    }
                } else if (d.type == QDQ_Q6_K) {
                    const int c0 = lane_col0<QDQ_Q6_K>(lane);
                    const uint32_t xs = xbuf_a + 4 * (kind_off[kind] + xcol + c0);
                    if (256 * (lane >> 2) < cols_here) {
                        if (BT == 1 && (xr_epoch != st_epoch || xr_j != j || xr_type != d.type)) {
                            load_x<QDQ_Q6_K>(xs, 0, xr);
                            xr_epoch = st_epoch; xr_j = j; xr_type = d.type;
                        }
                        unit_q6k<BT>(wrow, lane, xr, xs, xstride, acc);
                    } else {
#pragma unroll
                        for (int b = 0; b < BT; ++b) acc.v[b] = 0.f;
                    }
                } else {
                    const int c0 = lane_col0<QDQ_Q8_0>(lane);
                    const uint32_t xs = xbuf_a + 4 * (kind_off[kind] + xcol + c0);
                    const int nblk = cols_here / 32;
                    if (2 * lane < nblk) {
                        if (BT == 1 && (xr_epoch != st_epoch || xr_j != j || xr_type != d.type)) {
                            load_x<QDQ_Q8_0>(xs, 0, xr);
                            xr_epoch = st_epoch; xr_j = j; xr_type = d.type;
                        }
                        if (d.type == QDQ_Q8_0) unit_q8_0<BT>(wrow, lane, nblk, xr, xs, xstride, acc);
                        else unit_q4_0<BT>(wrow, lane, nblk, xr, xs, xstride, acc);
                    } else {
#pragma unroll
                        for (int b = 0; b < BT; ++b) acc.v[b] = 0.f;
                    }
                }
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    const float v = warp_sum(acc.v[b]);
                    if (lane == 0) pbuf[u * BT + b] = v;
                }
            }
            named_bar_sync(1, kConsumers);
            if (ctid == 0) mbar_arrive(empty_a + 8 * s);
            // fixed-order sum over column blocks, then store
            for (int i = ctid; i < tl.nrows * BT; i += kConsumers) {
                const int r = i / BT, b = i - r * BT;
                if (b >= a.batch) continue;
                float sum = 0.f;
                for (int j = 0; j < geo.ncb; ++j) sum += pbuf[(j * tl.nrows + r) * BT + b];
                float *yp = d.y + (int64_t)b * d.rows + tl.row0 + r;
                if (tl.kc0 == 0) *yp = sum;
                else *yp += sum;
            }
            pb ^= 1;
            ++t;
        },
        [&](int L) {
            if (a.counters != nullptr) {
                named_bar_sync(1, kConsumers);  // this CTA's y stores of level L are done
                if (ctid == 0) {
                    __threadfence();
                    const unsigned old = atomicAdd(&a.counters[L], 1u);
                    if (L == a.nlevels - 1 && old == (unsigned)P - 1) {
                        // every CTA has passed every wait: reset for the next run
                        for (int i = 0; i < a.nlevels; ++i) a.counters[i] = 0u;
                        __threadfence();
                    }
                }
            }
        });
}

__global__ void wait_selftest_kernel(const unsigned *flag, int64_t limit_ns) {
    wait_counter(flag, 1u, &s_status_stream, (uint64_t)limit_ns);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct StreamPlanHost {
    int bt;
    int grid;
    bool cooperative;
    size_t args_bytes;
    void *args;  // StreamArgs<...>
    bool big;
};

template <int MAXD, int MAXL>
static void fill_args(StreamArgs<MAXD, MAXL> *A, const qdq_gemv_desc *descs, const int *level, int n, int batch,
                      unsigned *counters, int BT) {
    memset(A, 0, sizeof(*A));
    A->ndesc = n;
    A->batch = batch;
    A->counters = counters;
    int L = 0;
    A->level_start[0] = 0;
    for (int i = 0; i < n; ++i) {
        const int lv = level ? level[i] : 0;
        while (L < lv) A->level_start[++L] = i;
    }
    A->nlevels = L + 1;
    A->level_start[L + 1] = n;
    for (int i = 0; i < n; ++i) {
        DevDesc &d = A->d[i];
        d.W = (const uint8_t *)descs[i].W;
        d.x = descs[i].x;
        d.y = descs[i].y;
        d.rows = descs[i].rows;
        d.cols = (int32_t)descs[i].cols;
        d.type = descs[i].type;
        d.rb = (int32_t)((descs[i].cols / blk_weights(d.type)) * blk_bytes(d.type));
    }
    // copy kinds per (level, x) and the column chunk
    for (int lv = 0; lv < A->nlevels; ++lv) {
        for (int i = A->level_start[lv]; i < A->level_start[lv + 1]; ++i) {
            int kinds = 0;
            for (int k = A->level_start[lv]; k < A->level_start[lv + 1]; ++k)
                if (A->d[k].x == A->d[i].x) kinds |= 1 << x_kind(A->d[k].type);
            A->d[i].kinds = kinds;
        }
    }
    const int xbytes = BT == 1 ? Cfg<1>::kXBytes : Cfg<8>::kXBytes;
    for (int i = 0; i < n; ++i) {
        DevDesc &d = A->d[i];
        const int ncopies = __builtin_popcount(d.kinds);
        int kc_x = xbytes / (4 * BT * ncopies);
        kc_x -= kc_x % 256;
        // a row segment of kc columns must fit one stage slot
        const int per256 = (256 / blk_weights(d.type)) * blk_bytes(d.type);
        int kc_w = ((kStageBytes - 32) / per256) * 256;
        int kc = kc_x < kc_w ? kc_x : kc_w;
        if (kc > kXSumFloats / BT * 32) kc = kXSumFloats / BT * 32;  // Q4_K sums fit their region
        if (kc >= d.cols) kc = d.cols;
        d.kc = kc;
    }
}

static int bt_of(int batch) { return batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }

template <int BT, int MAXD, int MAXL>
static int launch_typed(const StreamPlanHost *p, cudaStream_t stream) {
    auto kern = stream_kernel<BT, MAXD, MAXL>;
    static bool attr_done[16] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 15]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<BT>()) !=
            cudaSuccess)
            return QDQ_ERR_CUDA;
        attr_done[dev & 15] = true;
    }
    void *params[] = {p->args};
    cudaError_t e;
    if (p->cooperative)
        e = cudaLaunchCooperativeKernel((const void *)kern, dim3(p->grid), dim3(kThreads), params,
                                        (size_t)smem_bytes<BT>(), stream);
    else
        e = cudaLaunchKernel((const void *)kern, dim3(p->grid), dim3(kThreads), params, (size_t)smem_bytes<BT>(),
                             stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
}

int stream_plan_build(const qdq_gemv_desc *descs, const int *level, int n, int batch, unsigned *counters,
                      int sm_count, StreamPlanHost **out) {
    StreamPlanHost *p = new (std::nothrow) StreamPlanHost();
    if (!p) return QDQ_ERR_CUDA;
    p->bt = bt_of(batch);
    p->grid = sm_count;
    const int nlev = level ? level[n - 1] + 1 : 1;
    p->big = n > kMaxGroupDescs || nlev > 1;
    p->cooperative = nlev > 1;
    if (p->big) {
        using A = StreamArgs<kMaxPlanDescs, kMaxPlanLevels>;
        A *args = (A *)malloc(sizeof(A));
        if (!args) { delete p; return QDQ_ERR_CUDA; }
        fill_args(args, descs, level, n, batch, counters, p->bt);
        p->args = args;
        p->args_bytes = sizeof(A);
    } else {
        using A = StreamArgs<kMaxGroupDescs, 1>;
        A *args = (A *)malloc(sizeof(A));
        if (!args) { delete p; return QDQ_ERR_CUDA; }
        fill_args(args, descs, level, n, batch, counters, p->bt);
        p->args = args;
        p->args_bytes = sizeof(A);
    }
    *out = p;
    return QDQ_OK;
}

int stream_plan_launch(const StreamPlanHost *p, cudaStream_t stream) {
    if (p->big) {
        switch (p->bt) {
            case 1: return launch_typed<1, kMaxPlanDescs, kMaxPlanLevels>(p, stream);
            case 2: return launch_typed<2, kMaxPlanDescs, kMaxPlanLevels>(p, stream);
            case 4: return launch_typed<4, kMaxPlanDescs, kMaxPlanLevels>(p, stream);
            default: return launch_typed<8, kMaxPlanDescs, kMaxPlanLevels>(p, stream);
        }
    }
    switch (p->bt) {
        case 1: return launch_typed<1, kMaxGroupDescs, 1>(p, stream);
        case 2: return launch_typed<2, kMaxGroupDescs, 1>(p, stream);
        case 4: return launch_typed<4, kMaxGroupDescs, 1>(p, stream);
        default: return launch_typed<8, kMaxGroupDescs, 1>(p, stream);
    }
}

// Multi-level launch with caller-provided level counters and no heap use: the
// kernel arguments live on this function's stack (about 10 KiB).
int stream_launch_levels_inplace(const qdq_gemv_desc *descs, const int *level, int n, int batch,
                                 unsigned *counters, int sm_count, cudaStream_t stream) {
    using A = StreamArgs<kMaxPlanDescs, kMaxPlanLevels>;
    A args;
    StreamPlanHost p;
    p.bt = bt_of(batch);
    p.grid = sm_count;
    p.big = true;
    p.cooperative = true;
    p.args = &args;
    p.args_bytes = sizeof(A);
    fill_args(&args, descs, level, n, batch, counters, p.bt);
    return stream_plan_launch(&p, stream);
}

void stream_plan_free(StreamPlanHost *p) {
    if (!p) return;
    free(p->args);
    delete p;
}

int stream_plan_nlevels(const StreamPlanHost *p) {
    return p->big ? ((StreamArgs<kMaxPlanDescs, kMaxPlanLevels> *)p->args)->nlevels : 1;
}

int take_status_stream() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, s_status_stream, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(s_status_stream, &zero, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    return v;
}

int launch_wait_selftest(int64_t limit_ns, cudaStream_t stream) {
    unsigned *flag = nullptr;
    if (cudaMallocAsync((void **)&flag, sizeof(unsigned), stream) != cudaSuccess) return QDQ_ERR_CUDA;
    cudaMemsetAsync(flag, 0, sizeof(unsigned), stream);
    wait_selftest_kernel<<<1, 1, 0, stream>>>(flag, limit_ns);
    const cudaError_t e = cudaGetLastError();
    cudaFreeAsync(flag, stream);
    return e == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

}  // namespace qdq
