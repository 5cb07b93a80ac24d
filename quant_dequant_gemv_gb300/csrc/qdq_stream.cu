// qdq_stream.cu -- fused dequant-GEMV on CUDA cores, batch 1..8.
//
// "S21 The Capstone: picoLM, in Python", section 3 (fused dequant + dot: walk
// the quantised bytes and accumulate the dot product while decoding, so only
// the 4-bit data crosses the memory bus) and section 4 (model_forward: the
// per-layer projections of a decode step); "PETIT" (gemv_q8 / gemv_q4, weights
// stored out x in).
//
// One persistent CTA per SM, warp-specialised:
//  * Work: GEMVs in dependency levels. In each level the level's rows are split
//    across CTAs by weight bytes (each CTA's row ranges are computed once, into
//    shared memory). A CTA walks its rows in tiles of whole rows (or row
//    segments of a column chunk) that fit one 32 KiB shared-memory stage.
//  * Warp 0, the producer, streams tile bytes HBM -> shared memory with 1-D bulk
//    copies (cp.async.bulk, no multicast) into a ring of stages (full/empty
//    mbarriers). It never waits for level dependencies: weights do not depend on
//    earlier outputs, so it fetches ahead into later levels.
//  * Warp 1, the control warp, owns the level dependency: when this CTA's
//    consumers finish level L it publishes that (one global counter per level)
//    and waits until every CTA has; then it stages the next input x into one of
//    two x slots (plain, and pre-scaled copies for the nibble formats, plus the
//    Q4_K sub-block sums of x) and releases it to the consumers.
//  * Warps 2..9, the consumers, each own whole rows (row index mod 8): a lane
//    covers 64 weights of a 2048-column block; for batch 1 its x values stay in
//    registers across rows. Nibbles and 6-bit quants become floats by
//    exponent-field construction, products accumulate in packed f32x2 FMAs, and
//    one warp shuffle tree per row gives y, written by the owning warp. There is
//    no CTA-wide barrier on the data path: warps release stages and x slots
//    through mbarriers with one arrival per warp.
//  * Every wait is bounded (qdq_device.cuh).
#include <cstdio>
#include <cstring>
#include <new>
#include <type_traits>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {

static __device__ int s_status_stream;

// Phase timestamps for performance analysis, compiled in only with -DQDQ_TRACE:
// trace[(cta * nlevels + level) * 16 + slot] = %globaltimer.
#ifdef QDQ_TRACE
#define QDQ_TR(L, slot)                                                                                 \
    do {                                                                                                \
        if (a.trace) a.trace[((size_t)blockIdx.x * a.nlevels + (L)) * 16 + (slot)] = globaltimer_ns(); \
    } while (0)
#else
#define QDQ_TR(L, slot) \
    do {                \
    } while (0)
#endif

constexpr int kConsumerWarps = 8;
constexpr int kFirstConsumerWarp = 2;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = 32 * (kConsumerWarps + kFirstConsumerWarp);
constexpr int kStageBytes = 32768;
constexpr int kCB = 2048;  // columns per column block (32 lanes x 64)

template <int BT> struct Cfg;
// kStages: ring depth; kXBytes / kXSumBytes: one x slot (there are two)
template <> struct Cfg<1> { static constexpr int kStages = 5, kXBytes = 24576, kXSumBytes = 1024; };
template <> struct Cfg<2> { static constexpr int kStages = 4, kXBytes = 40960, kXSumBytes = 2048; };
template <> struct Cfg<4> { static constexpr int kStages = 4, kXBytes = 40960, kXSumBytes = 2048; };
template <> struct Cfg<8> { static constexpr int kStages = 4, kXBytes = 40960, kXSumBytes = 2048; };

struct DevDesc {
    const uint8_t *W;
    const float *x;
    float *y;
    int64_t rows;
    int32_t cols;
    int32_t type;
    int32_t rb;     // bytes per row
    int32_t kc;     // columns per x chunk
    int32_t kinds;  // bit k: the level's x needs swizzled copy kind k (0 plain, 1 Q4_K-scaled, 2 q4_0-scaled)
    int32_t pad;
};

template <int MAXD, int MAXL>
struct StreamArgs {
    int32_t ndesc, nlevels, batch, pad;
    unsigned *counters;
    unsigned long long *trace;  // QDQ_TRACE builds only: per-CTA phase timestamps
    int32_t level_start[MAXL + 1];
    DevDesc d[MAXD];
};

template <int BT, int MAXD>
constexpr int smem_bytes() {
    return Cfg<BT>::kStages * kStageBytes + 2 * Cfg<BT>::kXBytes + 2 * Cfg<BT>::kXSumBytes + MAXD * 16 +
           (2 * Cfg<BT>::kStages + 6) * 8;
}

// ---------------------------------------------------------------------------
// Format constants
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int blk_bytes(int t) {
    return t == QDQ_Q4_K ? 144 : t == QDQ_Q6_K ? 210 : t == QDQ_Q8_0 ? 36 : 18;
}
__host__ __device__ constexpr int blk_weights(int t) { return (t == QDQ_Q4_K || t == QDQ_Q6_K) ? 256 : 32; }
__host__ __device__ constexpr int x_kind(int t) { return t == QDQ_Q4_K ? 1 : t == QDQ_Q4_0 ? 2 : 0; }

// Float offsets inside an x slot: the swizzled copies in kind order, each
// [batch][kc] floats.
QDQ_DEV int copy_offset(int kinds, int kind, int kc, int BT) {
    int off = 0;
    for (int k = 0; k < kind; ++k)
        if ((kinds >> k) & 1) off += kc * BT;
    return off;
}

// Swizzled x layout: the 16-byte chunk c of a staged row is stored at chunk
// c ^ rev3((c >> 4) & 7). Lanes read 64-float runs at 256-byte strides (Q4_K,
// q8_0, q4_0) or 16-float runs at 64/512/1024-byte offsets (Q6_K); with the
// swizzle the eight lanes of each quarter-warp hit eight different bank groups.
QDQ_DEV int xswz(int c) {
    const int v = (c >> 4) & 7;
    return c ^ (((v & 1) << 2) | (v & 2) | (v >> 2));
}
// Four floats at logical offset `off` (a multiple of 4) of a swizzled row.
QDQ_DEV uint4 xload4(const float *row, int off) { return *(const uint4 *)(row + 4 * xswz(off >> 2)); }

// ---------------------------------------------------------------------------
// The schedule: identical for the producer, the control warp and the consumers.
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
    t.rmax = contiguous ? (kStageBytes - 32) / d.rb : kStageBytes / t.pitch;
    if (t.rmax < 1) t.rmax = 1;
    return t;
}

// Rows [ra, rb) of desc g that CTA `cta` owns in its level (byte-balanced split).
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
        const int64_t off = byte - start;
        if (off <= 0) return 0;
        const int64_t r = (off + rbytes - 1) / rbytes;
        return r < rows ? r : rows;
    };
    *ra = row_at(A0);
    *rb = row_at(B0);
}

// Calls on_begin(L) / on_end(L) around each level and on_tile(tile, geom, epoch,
// new_epoch, desc) for every tile. An epoch is one staged x: (level, x buffer,
// chunk).
template <class A, class FBegin, class FTile, class FEnd>
QDQ_DEV void walk(const A &a, const int64_t *ranges, FBegin &&on_begin, FTile &&on_tile, FEnd &&on_end) {
    int epoch = -1;
    for (int L = 0; L < a.nlevels; ++L) {
        on_begin(L);
        const float *ex = nullptr;
        int ekc = -1;
        const int g_end = a.level_start[L + 1];
        for (int g = a.level_start[L]; g < g_end; ++g) {
            const int64_t ra = ranges[2 * g], rb = ranges[2 * g + 1];
            if (ra >= rb) continue;
            const DevDesc d = a.d[g];  // one read of the descriptor per GEMV, into registers
            for (int kc0 = 0; kc0 < d.cols; kc0 += d.kc) {
                const int kcols = d.cols - kc0 < d.kc ? d.cols - kc0 : d.kc;
                const bool contiguous = (kc0 == 0 && kcols == d.cols);
                const TileGeom geo = tile_geom(d, kcols, contiguous);
                const bool fresh = (d.x != ex || kc0 != ekc);
                if (fresh) {
                    ++epoch;
                    ex = d.x;
                    ekc = kc0;
                }
                bool first = fresh;
                for (int64_t r0 = ra; r0 < rb; r0 += geo.rmax) {
                    Tile t;
                    t.g = g;
                    t.row0 = r0;
                    t.nrows = (int)(rb - r0 < geo.rmax ? rb - r0 : geo.rmax);
                    t.kc0 = kc0;
                    t.kcols = kcols;
                    t.contiguous = contiguous;
                    on_tile(t, geo, epoch, first, d);
                    first = false;
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

QDQ_DEV uint32_t tile_bytes(const DevDesc &d, const Tile &t, const TileGeom &geo, uint32_t stage, uint32_t bar,
                            int mode) {
    const uint8_t *w_end = d.W + d.rows * (int64_t)d.rb;
    if (t.contiguous) return copy_span(d.W + t.row0 * d.rb, (uint32_t)t.nrows * d.rb, w_end, stage, bar, mode);
    uint32_t total = 0;
    const int64_t off = (int64_t)(t.kc0 / blk_weights(d.type)) * blk_bytes(d.type);
    for (int r = 0; r < t.nrows; ++r)
        total += copy_span(d.W + (t.row0 + r) * d.rb + off, (uint32_t)geo.segbytes, w_end,
                           stage + (uint32_t)(r * geo.pitch), bar, mode);
    return total;
}

// Shared-memory address of a row's segment in a stage.
QDQ_DEV uint32_t row_addr(const DevDesc &d, const Tile &t, const TileGeom &geo, uint32_t stage, int64_t row) {
    const int r = (int)(row - t.row0);
    if (t.contiguous) return stage + (uint32_t)((uintptr_t)(d.W + t.row0 * d.rb) & 15) + (uint32_t)r * d.rb;
    const int64_t off = (int64_t)(t.kc0 / blk_weights(d.type)) * blk_bytes(d.type);
    return stage + (uint32_t)r * geo.pitch + (uint32_t)((uintptr_t)(d.W + row * d.rb + off) & 15);
}

// ---------------------------------------------------------------------------
// Consumer: per-format work on NR rows x one column block.
//   wrow[r]: first byte of this column block in row r (shared memory).
//   xr:      batch 1: the lane's 64 x values as 32 float pairs (pre-scaled for
//            the nibble formats) and, for Q4_K, the sums of x over its two
//            sub-blocks; shared by the NR rows.
//   xs:      batch > 1 (NR = 1): the lane's x slice for batch 0 in the matching
//            staged copy; batch b is at xs + b * xstride floats.
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

QDQ_DEV void load_pairs16(const float *row, int off, uint64_t *dst) {  // 16 floats -> 8 pairs
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = xload4(row, off + 4 * i);
        dst[2 * i] = bits2(v.x, v.y);
        dst[2 * i + 1] = bits2(v.z, v.w);
    }
}

template <int TYPE>
QDQ_DEV int lane_col0(int lane) {
    if constexpr (TYPE == QDQ_Q4_K) return 256 * (lane >> 2) + 64 * (lane & 3);
    else if constexpr (TYPE == QDQ_Q6_K) return 256 * (lane >> 2) + 128 * ((lane >> 1) & 1) + 16 * (lane & 1);
    else return 64 * lane;
}

template <int TYPE>
QDQ_DEV void load_x(const float *xrow, int off, const float *xsum, XSlice &x) {
    if constexpr (TYPE == QDQ_Q6_K) {  // four runs of 16 at stride 32
#pragma unroll
        for (int k = 0; k < 4; ++k) load_pairs16(xrow, off + 32 * k, &x.v[8 * k]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) load_pairs16(xrow, off + 16 * k, &x.v[8 * k]);
    }
    if constexpr (TYPE == QDQ_Q4_K) {
        x.s0 = xsum[0];
        x.s1 = xsum[1];
    }
}

QDQ_DEV uint64_t pairsum_zero() { return 0; }

// Q4_K: lane = 4 s + c covers chunk c of super-block s: sub-block 2c (low nibbles,
// x[0..31] of the slice) and 2c+1 (high nibbles, x[32..63]).
// sum = d * (sc_lo * sum(q x)_lo + sc_hi * sum(q x)_hi) - dmin * (mn_lo * sum(x)_lo + mn_hi * sum(x)_hi)
template <int BT, int NR>
QDQ_DEV void unit_q4k(const uint8_t *const *wrow, int lane, const XSlice &xr, const float *xrow, int xoff,
                      int xstride, const float *xsum, int xsum_stride, float (&out)[NR][BT]) {
    const int s = lane >> 2, c = lane & 3;
    uint4 H[NR], Qa[NR], Qb[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const uint8_t *sb = wrow[r] + 144 * s;
        H[r] = ld4(sb);
        Qa[r] = ld4(sb + 16 + 32 * c);
        Qb[r] = ld4(sb + 32 + 32 * c);
    }
    const uint64_t M2 = bits2(__float_as_uint(kTwo23), __float_as_uint(kTwo23));
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        uint32_t sc2, mn2;
        q4k_pair_fields(H[r].y, H[r].z, H[r].w, c, &sc2, &mn2);
        const float d = half_bits_to_float(H[r].x & 0xFFFF), dmin = half_bits_to_float(H[r].x >> 16);
        const float sc_lo = (float)(sc2 & 0xFF), sc_hi = (float)(sc2 >> 8);
        const float mn_lo = (float)(mn2 & 0xFF), mn_hi = (float)(mn2 >> 8);
        const uint32_t w[8] = {Qa[r].x, Qa[r].y, Qa[r].z, Qa[r].w, Qb[r].x, Qb[r].y, Qb[r].z, Qb[r].w};
        if constexpr (BT == 1) {
            uint64_t a0 = 0, a1 = 0, h0 = 0, h1 = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t v = w[t], u = v >> 16;
                a0 = ffma2(fsub2(bits2(mask_magic<0xFu>(v), mask_magic<0xF00u>(v)), M2), xr.v[2 * t], a0);
                a1 = ffma2(fsub2(bits2(mask_magic<0xF0000u>(v), mask_magic<0xF00u>(u)), M2), xr.v[2 * t + 1], a1);
                h0 = ffma2(fsub2(bits2(mask_magic<0xF0u>(v), mask_magic<0xF000u>(v)), M2), xr.v[16 + 2 * t], h0);
                h1 = ffma2(fsub2(bits2(mask_magic<0xF0u>(u), mask_magic<0xF000u>(u)), M2), xr.v[17 + 2 * t], h1);
            }
            const float lo = (lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1));
            const float hi = (lo_of(h0) + hi_of(h0)) + (lo_of(h1) + hi_of(h1));
            out[r][0] = d * (sc_lo * lo + sc_hi * hi) - dmin * (mn_lo * xr.s0 + mn_hi * xr.s1);
        } else {
            uint64_t q[32];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t v = w[t], u = v >> 16;
                q[2 * t] = fsub2(bits2(mask_magic<0xFu>(v), mask_magic<0xF00u>(v)), M2);
                q[2 * t + 1] = fsub2(bits2(mask_magic<0xF0000u>(v), mask_magic<0xF00u>(u)), M2);
                q[16 + 2 * t] = fsub2(bits2(mask_magic<0xF0u>(v), mask_magic<0xF000u>(v)), M2);
                q[17 + 2 * t] = fsub2(bits2(mask_magic<0xF0u>(u), mask_magic<0xF000u>(u)), M2);
            }
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                const float *xb = xrow + b * xstride;
                uint64_t a0 = 0, a1 = 0, h0 = 0, h1 = 0;
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const uint4 xl = xload4(xb, xoff + 2 * i), xh = xload4(xb, xoff + 32 + 2 * i);
                    a0 = ffma2(q[i], bits2(xl.x, xl.y), a0);
                    a1 = ffma2(q[i + 1], bits2(xl.z, xl.w), a1);
                    h0 = ffma2(q[16 + i], bits2(xh.x, xh.y), h0);
                    h1 = ffma2(q[17 + i], bits2(xh.z, xh.w), h1);
                }
                const float lo = (lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1));
                const float hi = (lo_of(h0) + hi_of(h0)) + (lo_of(h1) + hi_of(h1));
                const float s0 = xsum[b * xsum_stride], s1 = xsum[b * xsum_stride + 1];
                out[r][b] = d * (sc_lo * lo + sc_hi * hi) - dmin * (mn_lo * s0 + mn_hi * s1);
            }
        }
    }
}

// Q6_K: lane = 4 s + 2 h + m covers, in super-block s, half h and the 16-wide
// column group m of each of the four 32-runs k: elements 128h + 32k + 16m + l,
// l < 16, with scale scales[8h + 2k + m] (= element / 16).
template <int BT, int NR>
QDQ_DEV void unit_q6k(const uint8_t *const *wrow, int lane, const XSlice &xr, const float *xrow, int xoff,
                      int xstride, float (&out)[NR][BT]) {
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
        if constexpr (BT == 1) {
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint64_t a0 = 0, a1 = 0;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t b6 = q6k_quant_bytes((k & 1) ? ql1[r][t] : ql0[r][t], qh[r][t], k);
                    a0 = ffma2(fsub2(bits2(byte_to_magic<0>(b6), byte_to_magic<1>(b6)), M32), xr.v[8 * k + 2 * t], a0);
                    a1 = ffma2(fsub2(bits2(byte_to_magic<2>(b6), byte_to_magic<3>(b6)), M32), xr.v[8 * k + 2 * t + 1],
                               a1);
                }
                sum += sc[k] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
            }
            out[r][0] = d * sum;
        } else {
            uint64_t q[32];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t b6 = q6k_quant_bytes((k & 1) ? ql1[r][t] : ql0[r][t], qh[r][t], k);
                    q[8 * k + 2 * t] = fsub2(bits2(byte_to_magic<0>(b6), byte_to_magic<1>(b6)), M32);
                    q[8 * k + 2 * t + 1] = fsub2(bits2(byte_to_magic<2>(b6), byte_to_magic<3>(b6)), M32);
                }
            }
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                float sum = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float *xb = xrow + b * xstride;
                    uint64_t a0 = 0, a1 = 0;
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const uint4 xv = xload4(xb, xoff + 32 * k + 2 * i);
                        a0 = ffma2(q[8 * k + i], bits2(xv.x, xv.y), a0);
                        a1 = ffma2(q[8 * k + i + 1], bits2(xv.z, xv.w), a1);
                    }
                    sum += sc[k] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
                }
                out[r][b] = d * sum;
            }
        }
    }
}

// q8_0: lane covers blocks 2*lane and 2*lane+1 of the column block (x[0..31],
// x[32..63] of the slice). An int8 q becomes 2^23 + (q + 128) by flipping its
// sign bit and placing the byte under the exponent; subtracting 2^23 + 128
// leaves q exactly.
template <int BT, int NR>
QDQ_DEV void unit_q8_0(const uint8_t *const *wrow, int lane, int nblk_valid, const XSlice &xr, const float *xrow,
                       int xoff, int xstride, float (&out)[NR][BT]) {
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
                    const float *xb = xrow + b * xstride;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const uint4 xv = xload4(xb, xoff + 32 * i + 2 * j);
                        a0 = ffma2(q[16 * i + j], bits2(xv.x, xv.y), a0);
                        a1 = ffma2(q[16 * i + j + 1], bits2(xv.z, xv.w), a1);
                    }
                }
                sum += d[i] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
            }
            out[r][b] = sum;
        }
    }
}

// q4_0: lane covers blocks 2*lane, 2*lane+1 (36 bytes, 2-byte aligned). Byte i
// of a block holds weight i (low nibble) and weight i+16 (high nibble). Nibbles
// stay at their bit position p (x pre-scaled by 2^-p); subtracting 2^23 + 8*2^p
// gives (q - 8) * 2^p exactly.
template <int BT, int NR>
QDQ_DEV void unit_q4_0(const uint8_t *const *wrow, int lane, int nblk_valid, const XSlice &xr, const float *xrow,
                       int xoff, int xstride, float (&out)[NR][BT]) {
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
                    const float *xb = xrow + b * xstride;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const uint4 xv = xload4(xb, xoff + 32 * i + 2 * j);
                        a0 = ffma2(q[16 * i + j], bits2(xv.x, xv.y), a0);
                        a1 = ffma2(q[16 * i + j + 1], bits2(xv.z, xv.w), a1);
                    }
                }
                sum += d[i] * ((lo_of(a0) + hi_of(a0)) + (lo_of(a1) + hi_of(a1)));
            }
            out[r][b] = sum;
        }
    }
}

QDQ_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sums of a over lanes and of b over lanes in one tree: afterwards lane 0 holds
// sum(a) and lane 16 holds sum(b).
QDQ_DEV float warp_sum2(float a, float b, int lane) {
    const bool upper = lane & 16;
    float keep = upper ? b : a;
    const float send = upper ? a : b;
    keep += __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    return keep;
}

// Scale that puts x next to a nibble read at its bit position (see unit_q4k /
// unit_q4_0): low nibbles of bytes 0..3 of a word sit at bits 0, 8, 16, 8 (the
// last after a 16-bit shift), high nibbles at bits 4, 12, 4, 12.
QDQ_DEV float nibble_scale(bool high, int p) {
    const float lo = p == 0 ? 1.f : p == 2 ? 1.52587890625e-05f : 0.00390625f;
    const float hi = (p & 1) ? 0.000244140625f : 0.0625f;
    return high ? hi : lo;
}

// NR rows x one column block for the desc's format, into out (zero where the
// lane has nothing in this block).
template <int BT, int NR>
QDQ_DEV void run_unit(int type, const uint8_t *const *wrow, int lane, int cols_here, const XSlice &xr,
                      const float *xrow, int xoff, int xstride, const float *xsum, int xsum_stride,
                      float (&out)[NR][BT]) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) out[r][b] = 0.f;
    if (type == QDQ_Q4_K) {
        if (256 * (lane >> 2) < cols_here)
            unit_q4k<BT, NR>(wrow, lane, xr, xrow, xoff, xstride, xsum, xsum_stride, out);
    } else if (type == QDQ_Q6_K) {
        if (256 * (lane >> 2) < cols_here) unit_q6k<BT, NR>(wrow, lane, xr, xrow, xoff, xstride, out);
    } else {
        const int nblk = cols_here / 32;
        if (2 * lane < nblk) {
            if (type == QDQ_Q8_0) unit_q8_0<BT, NR>(wrow, lane, nblk, xr, xrow, xoff, xstride, out);
            else unit_q4_0<BT, NR>(wrow, lane, nblk, xr, xrow, xoff, xstride, out);
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int BT, int MAXD, int MAXL>
__global__ void __launch_bounds__(kThreads, 1)
    stream_kernel(const __grid_constant__ StreamArgs<MAXD, MAXL> a) {
    constexpr int NST = Cfg<BT>::kStages;
    constexpr int XB = Cfg<BT>::kXBytes, XSB = Cfg<BT>::kXSumBytes;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *ring = smem;
    uint8_t *xslot = smem + NST * kStageBytes;  // two slots of XB bytes
    uint8_t *xsum = xslot + 2 * XB;             // two slots of XSB bytes
    int64_t *ranges = (int64_t *)(xsum + 2 * XSB);
    uint64_t *bars = (uint64_t *)(ranges + 2 * MAXD);
    const uint32_t ring_a = smem_u32(ring), xslot_a = smem_u32(xslot), xsum_a = smem_u32(xsum);
    const uint32_t full_a = smem_u32(bars), empty_a = full_a + 8 * NST;
    // xready[2]: x slot staged (8 warp arrivals); xempty[2]: slot no longer read;
    // lvl: this CTA's consumers finished a level; dep: all CTAs finished the
    // previous level (arrival by the control warp).
    const uint32_t xready_a = empty_a + 8 * NST, xempty_a = xready_a + 16, lvl_a = xempty_a + 16;
    const uint32_t dep_a = lvl_a + 8;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, P = gridDim.x;
    int *status = &s_status_stream;
    const bool levels_synced = a.counters != nullptr;
    const int batch = a.batch;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full_a + 8 * s, 1);
            mbar_init(empty_a + 8 * s, kConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(xready_a + 8 * b, kConsumerWarps);
            mbar_init(xempty_a + 8 * b, kConsumerWarps);
        }
        mbar_init(lvl_a, kConsumerWarps);
        mbar_init(dep_a, 1);
        fence_mbar_init();
    }
    // this CTA's row range of every GEMV
    for (int L = 0; L < a.nlevels; ++L)
        for (int g = a.level_start[L] + (int)threadIdx.x; g < a.level_start[L + 1]; g += kThreads)
            cta_rows(a, L, g, cta, P, &ranges[2 * g], &ranges[2 * g + 1]);
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        int t = 0;
        walk(
            a, ranges, [](int) {},
            [&](const Tile &tl, const TileGeom &geo, int, bool, const DevDesc &d) {
                const int s = t % NST;
                if (t >= NST) mbar_wait(empty_a + 8 * s, ((t / NST) + 1) & 1, status);
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

    if (warp == 1) {
        // ------------------------------------------------------------ control
        // Publishes level L once this CTA's consumers have finished it, then
        // waits until every CTA has, and releases the consumers into level L+1.
        // The level barrier completes one phase per level in which this CTA has
        // tiles (consumers arrive only then) and so does dep (arrived only for
        // levels with tiles): neither can run two phases ahead of its waiter,
        // since consumers reach a level's work only through dep and dep for a
        // later level needs this level's publication first.
        if (!levels_synced) return;
        auto has_tiles = [&](int L) {
            for (int g = a.level_start[L]; g < a.level_start[L + 1]; ++g)
                if (ranges[2 * g] < ranges[2 * g + 1]) return true;
            return false;
        };
        int lvl_phase = 0;
        bool prev_had = has_tiles(0);
        for (int L = 1; L < a.nlevels; ++L) {
            if (lane == 0) QDQ_TR(L, 0);
            if (prev_had) mbar_wait(lvl_a, (lvl_phase++) & 1, status);
            if (lane == 0) {
                QDQ_TR(L, 1);
                // Consumers' y stores are ordered before their arrivals on the level
                // barrier (CTA scope); the release makes them visible at GPU scope
                // together with the count.
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&a.counters[L - 1]) : "memory");
                wait_counter(&a.counters[L - 1], (unsigned)P, status, kWaitLimitNs);
                QDQ_TR(L, 2);
            }
            __syncwarp();
            const bool had = has_tiles(L);
            if (had && lane == 0) mbar_arrive(dep_a);
            prev_had = had;
        }
        if (prev_had) mbar_wait(lvl_a, (lvl_phase++) & 1, status);
        if (lane == 0) {
            __threadfence();
            const unsigned old = atomicAdd(&a.counters[a.nlevels - 1], 1u);
            if (old == (unsigned)P - 1) {
                // every CTA has passed every wait: reset for the next run
                for (int i = 0; i < a.nlevels; ++i) a.counters[i] = 0u;
                __threadfence();
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - kFirstConsumerWarp;
    const int ctid = (int)threadIdx.x - 32 * kFirstConsumerWarp;
    int t = 0, cur_e = -1, cur_level = 0, tiles_in_level = 0, dep_phase = 0;
    bool had_tiles = false, dep_pending = false;
    (void)cur_level;
    (void)tiles_in_level;
    XSlice xr;
    int xr_key = -1;  // (epoch, column block, format) of the x values in xr

    walk(
        a, ranges,
        [&](int L) {
            cur_level = L;
            tiles_in_level = 0;
            dep_pending = L > 0 && levels_synced;
        },
        [&](const Tile &tl, const TileGeom &geo, int e, bool, const DevDesc &d) {
            had_tiles = true;
            if (cw == 0 && lane == 0 && tiles_in_level == 0) QDQ_TR(cur_level, 4);
            if (e != cur_e) {
                if (cur_e >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xempty_a + 8 * (cur_e & 1));
                }
                if (dep_pending) {  // the previous level is complete on every CTA
                    mbar_wait(dep_a, (dep_phase++) & 1, status);
                    dep_pending = false;
                }
                cur_e = e;
                const int b = e & 1;
                if (e >= 2) mbar_wait(xempty_a + 8 * b, ((e >> 1) - 1) & 1, status);
                // Stage x[:, kc0 : kc0 + kcols] into slot b (every consumer thread a
                // share): swizzled plain and/or pre-scaled copies, and the Q4_K
                // sub-block sums of x. Loads bypass L1: x may have been written by
                // other SMs during this kernel.
                float *xs = (float *)(xslot + b * XB);
                float *xsm = (float *)(xsum + b * XSB);
                const int kc = tl.kcols, n4 = kc / 4;
                const bool k0 = d.kinds & 1, k1 = d.kinds & 2, k2 = d.kinds & 4;
                const int o0 = copy_offset(d.kinds, 0, kc, BT), o1 = copy_offset(d.kinds, 1, kc, BT),
                          o2 = copy_offset(d.kinds, 2, kc, BT);
#pragma unroll 4
                for (int i = ctid; i < n4 * BT; i += kConsumers) {
                    const int bb = i / n4, c = i - bb * n4, col = 4 * c;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (bb < batch) v = __ldcg((const float4 *)(d.x + (int64_t)bb * d.cols + tl.kc0) + c);
                    const int at = bb * kc + 4 * xswz(c);
                    if (k0) *(float4 *)(xs + o0 + at) = v;
                    if (k1) {  // Q4_K: low nibbles are columns 0..31 of each 64
                        const bool hi = (col & 63) >= 32;
                        *(float4 *)(xs + o1 + at) =
                            make_float4(v.x * nibble_scale(hi, 0), v.y * nibble_scale(hi, 1),
                                        v.z * nibble_scale(hi, 2), v.w * nibble_scale(hi, 3));
                        // sum of x over each 32-column sub-block: 8 lanes hold one sub-block
                        float sm = (v.x + v.y) + (v.z + v.w);
                        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
                        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
                        sm += __shfl_xor_sync(0xffffffffu, sm, 4);
                        if ((lane & 7) == 0) xsm[bb * (kc / 32) + col / 32] = sm;
                    }
                    if (k2) {  // q4_0: low nibbles are columns 0..15 of each 32
                        const bool hi = (col & 31) >= 16;
                        *(float4 *)(xs + o2 + at) =
                            make_float4(v.x * nibble_scale(hi, 0), v.y * nibble_scale(hi, 1),
                                        v.z * nibble_scale(hi, 2), v.w * nibble_scale(hi, 3));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xready_a + 8 * b);
                mbar_wait(xready_a + 8 * b, (e >> 1) & 1, status);
            }
            if (cw == 0 && lane == 0 && tiles_in_level == 0) QDQ_TR(cur_level, 5);
            const int s = t % NST;
            mbar_wait(full_a + 8 * s, (t / NST) & 1, status);
            if (cw == 0 && lane == 0 && tiles_in_level == 0) QDQ_TR(cur_level, 6);
            ++tiles_in_level;
            const uint32_t stage = ring_a + s * kStageBytes;
            const uint8_t *stage_p = ring + s * kStageBytes;
            const int qk = blk_weights(d.type), bb = blk_bytes(d.type);
            const int cb_bytes = (kCB / qk) * bb;
            const int kind = x_kind(d.type);
            const float *xcopy = (const float *)(xslot + (e & 1) * XB) + copy_offset(d.kinds, kind, tl.kcols, BT);
            const float *xsum_base = (const float *)(xsum + (e & 1) * XSB);
            const int xstride = tl.kcols, xss = tl.kcols / 32;
            const int c0 = d.type == QDQ_Q4_K ? lane_col0<QDQ_Q4_K>(lane)
                           : d.type == QDQ_Q6_K ? lane_col0<QDQ_Q6_K>(lane)
                                                : lane_col0<QDQ_Q8_0>(lane);
            const int64_t end = tl.row0 + tl.nrows;
            // rows of this tile owned by this warp: row index = cw (mod 8)
            int64_t row = tl.row0 + ((cw - (int)(tl.row0 % kConsumerWarps) + kConsumerWarps) % kConsumerWarps);
            // NR rows (row, row + 8) x all column blocks of this chunk -> y
            auto process = [&](auto nr_tag, int64_t row_a) {
                constexpr int NR = decltype(nr_tag)::value;
                const uint8_t *wbase[NR];
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    wbase[r] = stage_p + (row_addr(d, tl, geo, stage, row_a + r * kConsumerWarps) - stage);
                float tot[NR][BT];
#pragma unroll
                for (int r = 0; r < NR; ++r)
#pragma unroll
                    for (int b = 0; b < BT; ++b) tot[r][b] = 0.f;
                for (int j = 0; j < geo.ncb; ++j) {
                    const int cols_here = tl.kcols - j * kCB < kCB ? tl.kcols - j * kCB : kCB;
                    const int xoff = j * kCB + c0;  // logical offset of the lane's slice in the row
                    const float *xsa = xsum_base + (j * kCB + c0) / 32;
                    if constexpr (BT == 1) {
                        const int key = (e * 64 + j) * 8 + d.type;
                        if (key != xr_key) {
                            const bool lane_live = (d.type == QDQ_Q8_0 || d.type == QDQ_Q4_0)
                                                       ? 64 * lane < cols_here
                                                       : 256 * (lane >> 2) < cols_here;
                            if (lane_live) {
                                if (d.type == QDQ_Q4_K) load_x<QDQ_Q4_K>(xcopy, xoff, xsa, xr);
                                else if (d.type == QDQ_Q6_K) load_x<QDQ_Q6_K>(xcopy, xoff, xsa, xr);
                                else load_x<QDQ_Q8_0>(xcopy, xoff, xsa, xr);
                            }
                            xr_key = key;
                        }
                    }
                    const uint8_t *wj[NR];
#pragma unroll
                    for (int r = 0; r < NR; ++r) wj[r] = wbase[r] + j * cb_bytes;
                    float acc[NR][BT];
                    run_unit<BT, NR>(d.type, wj, lane, cols_here, xr, xcopy, xoff, xstride, xsa, xss, acc);
#pragma unroll
                    for (int r = 0; r < NR; ++r)
#pragma unroll
                        for (int b = 0; b < BT; ++b) tot[r][b] += acc[r][b];
                }
                if constexpr (NR == 2) {
                    const float v = warp_sum2(tot[0][0], tot[1][0], lane);
                    if (lane == 0 || lane == 16) {
                        float *yp = d.y + (lane == 0 ? row_a : row_a + kConsumerWarps);
                        if (tl.kc0 == 0) *yp = v;
                        else *yp += v;  // the same warp wrote the earlier chunks of this row
                    }
                } else {
#pragma unroll
                    for (int b = 0; b < BT; ++b) {
                        const float v = warp_sum(tot[0][b]);
                        if (lane == 0 && b < batch) {
                            float *yp = d.y + (int64_t)b * d.rows + row_a;
                            if (tl.kc0 == 0) *yp = v;
                            else *yp += v;  // the same warp wrote the earlier chunks of this row
                        }
                    }
                }
            };
            if constexpr (BT == 1) {  // two rows at a time share the x registers
                for (; row + kConsumerWarps < end; row += 2 * kConsumerWarps)
                    process(std::integral_constant<int, 2>{}, row);
                if (row < end) process(std::integral_constant<int, 1>{}, row);
            } else {
                for (; row < end; row += kConsumerWarps) process(std::integral_constant<int, 1>{}, row);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_a + 8 * s);
            ++t;
        },
        [&](int) {
            if (cw == 0 && lane == 0) QDQ_TR(cur_level, 7);
            if (levels_synced && had_tiles) {
                __syncwarp();
                if (lane == 0) mbar_arrive(lvl_a);  // release (CTA scope) of this warp's y stores
            }
            had_tiles = false;
            dep_pending = false;  // a level without tiles here needs no release
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

#ifdef QDQ_TRACE
static unsigned long long *s_trace = nullptr;
#endif

static int xbytes_of(int BT) { return BT == 1 ? Cfg<1>::kXBytes : Cfg<8>::kXBytes; }
static int xsumbytes_of(int BT) { return BT == 1 ? Cfg<1>::kXSumBytes : Cfg<8>::kXSumBytes; }

template <int MAXD, int MAXL>
static void fill_args(StreamArgs<MAXD, MAXL> *A, const qdq_gemv_desc *descs, const int *level, int n, int batch,
                      unsigned *counters, int BT) {
    memset(A, 0, sizeof(*A));
#ifdef QDQ_TRACE
    A->trace = s_trace;
#endif
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
    // staged copy kinds per (level, x), and the column chunk
    for (int lv = 0; lv < A->nlevels; ++lv) {
        for (int i = A->level_start[lv]; i < A->level_start[lv + 1]; ++i) {
            int kinds = 0;
            for (int k = A->level_start[lv]; k < A->level_start[lv + 1]; ++k)
                if (A->d[k].x == A->d[i].x) kinds |= 1 << x_kind(A->d[k].type);
            A->d[i].kinds = kinds;
        }
    }
    for (int i = 0; i < n; ++i) {
        DevDesc &d = A->d[i];
        const int nregions = __builtin_popcount(d.kinds);  // swizzled copies
        int kc_x = xbytes_of(BT) / (4 * BT * nregions);
        const int kc_s = (xsumbytes_of(BT) / (4 * BT)) * 32;  // Q4_K sums fit their slot
        if (kc_s < kc_x) kc_x = kc_s;
        kc_x -= kc_x % 256;
        // a row segment of kc columns must fit one stage slot
        const int per256 = (256 / blk_weights(d.type)) * blk_bytes(d.type);
        const int kc_w = ((kStageBytes - 32) / per256) * 256;
        int kc = kc_x < kc_w ? kc_x : kc_w;
        if (kc >= d.cols) kc = d.cols;
        d.kc = kc;
    }
    // GEMVs of a level that share x must use the same chunking
    for (int lv = 0; lv < A->nlevels; ++lv)
        for (int i = A->level_start[lv]; i < A->level_start[lv + 1]; ++i)
            for (int k = A->level_start[lv]; k < i; ++k)
                if (A->d[k].x == A->d[i].x && A->d[k].kc < A->d[i].kc) A->d[i].kc = A->d[k].kc;
}

static int bt_of(int batch) { return batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }

template <int BT, int MAXD, int MAXL>
static int launch_typed(const StreamPlanHost *p, cudaStream_t stream) {
    auto kern = stream_kernel<BT, MAXD, MAXL>;
    RelaxedCaptureScope relaxed;  // the first launch sets the kernel's attributes
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 63]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<BT, MAXD>()) !=
            cudaSuccess) {
            cudaGetLastError();
            return QDQ_ERR_CUDA;
        }
        attr_done[dev & 63] = true;
    }
    void *params[] = {p->args};
    cudaError_t e;
    if (p->cooperative)
        e = cudaLaunchCooperativeKernel((const void *)kern, dim3(p->grid), dim3(kThreads), params,
                                        (size_t)smem_bytes<BT, MAXD>(), stream);
    else
        e = cudaLaunchKernel((const void *)kern, dim3(p->grid), dim3(kThreads), params,
                             (size_t)smem_bytes<BT, MAXD>(), stream);
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

#ifdef QDQ_TRACE
}  // namespace qdq
extern "C" void qdq_debug_set_trace(unsigned long long *buf) { qdq::s_trace = buf; }
namespace qdq {
#endif

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
