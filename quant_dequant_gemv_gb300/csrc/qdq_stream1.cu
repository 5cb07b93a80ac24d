// qdq_stream1.cu -- fused dequant-GEMV on CUDA cores for one input vector
// (batch 1): single GEMVs, groups and multi-level plans such as a decode step.
//
// "S21 The Capstone: picoLM, in Python", section 3 (fused dequant + dot: only the
// quantised bytes cross the memory bus, decoded in registers into the dot
// product) and section 4 (the per-layer projections of a decode step, each level
// waiting for the previous one); "PETIT" (gemv_q8 / gemv_q4, rows of 32-weight
// blocks, weights stored out x in).
//
// One persistent CTA per SM, warp-specialised, with the reduction dimension
// split across the consumer warps:
//  * A tile is up to 16 rows x one 2048-column chunk of a GEMV. Consumer warp w
//    owns the 256-column slice w of the chunk (one Q4_K / Q6_K super-block, eight
//    q8_0 / q4_0 blocks) for every row of the tile: lane 4 r + c covers rows r
//    and r + 8 and quarter c of the slice, 64 weights per row. Every warp works
//    on every row, so even a level with a dozen rows per CTA keeps all eight
//    warps busy, and a warp needs the x values of its slice only.
//  * Each warp stages its own x slices (plain and/or pre-scaled copies, plus the
//    Q4_K sub-block sums of x) into a private shared-memory area, straight from
//    global memory once the level's inputs are ready: no CTA-wide x handshake.
//  * A warp keeps its row partials for the whole level in a shared-memory buffer
//    (the chunks of a row add up in place); at the end of the level (or when the
//    buffer is full) the consumer warps meet once, add the eight partials of
//    each row in warp order and store y.
//  * Warp 0 streams tiles HBM -> shared memory with 1-D bulk copies into a ring
//    of stages and fetches ahead across level boundaries (W does not depend on
//    x). Warp 1 owns the level dependency: one device-wide counter per level.
//  * Every wait is bounded (qdq_device.cuh).
#include <cstdio>
#include <type_traits>

#include "qdq_stream_common.cuh"

namespace qdq {

static __device__ int s_status_s1;

// Phase timestamps for performance analysis, compiled in only with -DQDQ_TRACE:
// trace[(cta * nlevels + level) * 32 + slot] = %globaltimer (S1_TR) or the SM's
// clock64 (S1_TRC, per-tile phases of the first consumer warp).
#ifdef QDQ_TRACE
#define S1_TR(L, slot)                                                                                  \
    do {                                                                                                \
        if (a.trace) a.trace[((size_t)blockIdx.x * a.nlevels + (L)) * 32 + (slot)] = globaltimer_ns(); \
    } while (0)
#define S1_TRC(L, slot)                                                                                     \
    do {                                                                                                    \
        if (a.trace) a.trace[((size_t)blockIdx.x * a.nlevels + (L)) * 32 + (slot)] = (uint64_t)clock64(); \
    } while (0)
#else
#define S1_TR(L, slot) \
    do {               \
    } while (0)
#define S1_TRC(L, slot) \
    do {                \
    } while (0)
#endif

namespace s1 {

constexpr int kCW = 8;                            // consumer warps
constexpr int kFirstCW = 2;                       // warp 0 producer, warp 1 control
constexpr int kThreads = 32 * (kCW + kFirstCW);
constexpr int kPassRows = 16;                     // rows of one pass (lanes cover r and r + 8)
constexpr int kTileRows = 64;                     // rows of a whole-row tile (up to four passes)
constexpr int kChunkRows = 16;                    // rows of a chunked tile
constexpr int kChunk = 2048;                      // columns of a chunk: kCW slices of kSlice
constexpr int kSlice = 256;
constexpr int kRingBytes = 172032;                // W ring: tiles packed in order, wrapping
constexpr int kMaxTileBytes = kRingBytes / 2;     // at least two tiles in flight
constexpr int kSlots = 8;                         // full/empty barrier pairs (tiles in the ring)
constexpr int kXFloats = 1024;                    // private x area of one consumer warp
constexpr int kBufRows = 512;                     // rows of the level partial buffer
constexpr int kFlushBar = 1;                      // named barrier of the consumer warps

// Shared memory layout (bytes). The ring starts at 0 (1024-aligned base).
template <int MAXD>
struct Smem {
    static constexpr int kX = kRingBytes;
    static constexpr int kPart = kX + kCW * kXFloats * 4;     // [warp][buffer row] partials
    static constexpr int kDst = kPart + kCW * kBufRows * 4;   // y address of each buffer row
    static constexpr int kRanges = kDst + kBufRows * 8;
    static constexpr int kRing = kRanges + 2 * MAXD * 8;      // producer: live tiles' ring ranges
    static constexpr int kBars = kRing + 2 * kSlots * 4;
    static constexpr int kBytes = kBars + (2 * kSlots + 2) * 8;
};
static_assert(Smem<kMaxPlanDescs>::kBytes <= 227 * 1024, "shared memory budget");

// ---------------------------------------------------------------------------
// Tiles: identical sequence for the producer, the control warp and consumers.
// A whole-row tile holds up to 64 complete rows (one contiguous bulk copy) and
// every chunk of their x; rows too long for 8 per stage are cut into 2048-column
// chunks of up to 16 rows, copied row segment by row segment.
// ---------------------------------------------------------------------------
struct Tile {
    int g;            // GEMV (desc index)
    int nrows;        // 1..64 (whole rows) or 1..16 (chunked)
    int64_t row0;
    int chunk;        // chunked: the 2048-column chunk; whole rows: 0
    int ccols;        // columns of the tile (whole rows: all of them)
    int xw0;          // first chunk of the staged x window (chunk - xw0 indexes it)
    int xwn;          // chunks in that window
    bool whole;       // complete rows, contiguous in the stage
    bool first;       // first chunk of this row group in the window
    bool last;        // last chunk of this row group in the window
    bool first_win;   // the window starts at column 0 (y is stored, not accumulated)
};

QDQ_DEV int nkinds(int kinds) { return __popc(kinds & 7); }
// x floats one warp stages per chunk: one 256-float slice per copy kind, plus the
// eight Q4_K sub-block sums.
QDQ_DEV int xfloats_per_chunk(int kinds) { return kSlice * nkinds(kinds) + ((kinds & 2) ? 8 : 0); }
QDQ_DEV int window_chunks(int kinds) {
    const int w = kXFloats / xfloats_per_chunk(kinds);
    return w < 1 ? 1 : w;
}
// Bytes of one row segment of a chunk, and the stage pitch of such segments.
QDQ_DEV int seg_bytes(const DevDesc &d, int ccols) { return (ccols / blk_weights(d.type)) * blk_bytes(d.type); }
QDQ_DEV int seg_pitch(int seg) { return ((seg + 15) & ~15) + 16; }
// Rows of a whole-row tile (a multiple of 8 up to 64), or 0 when fewer than 8
// rows fit a stage or the row's x does not fit one window.
QDQ_DEV int whole_rows(const DevDesc &d) {
    const int nch = (d.cols + kChunk - 1) / kChunk;
    const int cap = (kMaxTileBytes - 32) / d.rb;
    if (cap < 8 || nch > window_chunks(d.kinds)) return 0;
    return cap >= kTileRows ? kTileRows : cap & ~7;
}
QDQ_DEV int chunk_rows(const DevDesc &d) {
    const int cap = kMaxTileBytes / seg_pitch(seg_bytes(d, kChunk));
    return cap < kChunkRows ? (cap < 1 ? 1 : cap) : kChunkRows;
}

// Bytes a tile takes in the ring (copy_span may start up to 15 bytes before and
// end up to 15 bytes after the tile's rows; chunk segments sit at their pitch).
QDQ_DEV uint32_t tile_ring_bytes(const DevDesc &d, int nrows, bool whole, int ccols) {
    const uint32_t b = whole ? (uint32_t)(nrows * d.rb + 32) : (uint32_t)(nrows * seg_pitch(seg_bytes(d, ccols)));
    return (b + 127u) & ~127u;
}
// Next tile's offset in the ring: packed after the previous one, or at 0 when it
// would not fit before the end. Producer and consumers run the same sequence.
QDQ_DEV uint32_t ring_place(uint32_t &next, uint32_t bytes) {
    if (next + bytes > (uint32_t)kRingBytes) next = 0;
    const uint32_t o = next;
    next += bytes;
    return o;
}

// on_begin(L) / on_end(L) around each level; on_tile(tile, epoch, desc) for every
// tile. An epoch is one staged x window: (level, x, columns, window).
template <class A, class FBegin, class FTile, class FEnd>
QDQ_DEV void walk(const A &a, const int64_t *ranges, FBegin &&on_begin, FTile &&on_tile, FEnd &&on_end) {
    int epoch = -1;
    for (int L = 0; L < a.nlevels; ++L) {
        on_begin(L);
        const float *ex = nullptr;
        int ew = -1, ecols = -1;
        for (int g = a.level_start[L]; g < a.level_start[L + 1]; ++g) {
            const int64_t ra = ranges[2 * g], rb = ranges[2 * g + 1];
            if (ra >= rb) continue;
            const DevDesc d = a.d[g];
            const int nch = (d.cols + kChunk - 1) / kChunk;
            const int n = (int)(rb - ra);  // rows of one GEMV on one CTA
            const int wr = whole_rows(d);
            if (wr > 0) {
                if (d.x != ex || 0 != ew || d.cols != ecols) {
                    ++epoch;
                    ex = d.x;
                    ew = 0;
                    ecols = d.cols;
                }
                for (int r = 0; r < n; r += wr) {
                    Tile t;
                    t.g = g;
                    t.nrows = n - r < wr ? n - r : wr;
                    t.row0 = ra + r;
                    t.chunk = 0;
                    t.ccols = d.cols;
                    t.xw0 = 0;
                    t.xwn = nch;
                    t.whole = true;
                    t.first = t.last = t.first_win = true;
                    on_tile(t, epoch, d);
                }
                continue;
            }
            const int wmax = window_chunks(d.kinds);
            const int nrmax = chunk_rows(d);
            const int ntg = (n + nrmax - 1) / nrmax;
            const int nbase = n / ntg, nextra = n - nbase * ntg;
            for (int w0 = 0; w0 < nch; w0 += wmax) {
                const int w1 = nch < w0 + wmax ? nch : w0 + wmax;
                if (d.x != ex || w0 != ew || d.cols != ecols) {
                    ++epoch;
                    ex = d.x;
                    ew = w0;
                    ecols = d.cols;
                }
                int64_t r = ra;
                for (int tg = 0; tg < ntg; ++tg) {
                    const int nr = nbase + (tg < nextra ? 1 : 0);
                    for (int j = w0; j < w1; ++j) {
                        Tile t;
                        t.g = g;
                        t.nrows = nr;
                        t.row0 = r;
                        t.chunk = j;
                        t.ccols = d.cols - j * kChunk < kChunk ? d.cols - j * kChunk : kChunk;
                        t.xw0 = w0;
                        t.xwn = w1 - w0;
                        t.whole = false;
                        t.first = j == w0;
                        t.last = j == w1 - 1;
                        t.first_win = w0 == 0;
                        on_tile(t, epoch, d);
                    }
                    r += nr;
                }
            }
        }
        on_end(L);
    }
}

// Rows [ra, rb) of GEMV g that CTA `cta` owns in level L. The level's CTAs are
// dealt out to its GEMVs in proportion to their weight bytes (rounded CTA
// boundaries over the cumulative bytes), and each GEMV's rows are split evenly
// among its CTAs, so a CTA normally works on a single GEMV per level: one x
// format and as few tiles as possible. A GEMV too small to earn a CTA of its own
// goes whole to the CTA at its position.
template <class A>
QDQ_DEV void cta_rows_by_gemv(const A &a, int L, int g, int cta, int P, int64_t *ra, int64_t *rb) {
    int64_t total = 0, before = 0;
    for (int i = a.level_start[L]; i < a.level_start[L + 1]; ++i) {
        const int64_t bytes = a.d[i].rows * (int64_t)a.d[i].rb;
        if (i < g) before += bytes;
        total += bytes;
    }
    const int64_t mine = a.d[g].rows * (int64_t)a.d[g].rb, rows = a.d[g].rows;
    *ra = *rb = 0;
    if (total <= 0 || rows <= 0) return;
    const int c0 = (int)((before * P + total / 2) / total);
    const int c1 = (int)(((before + mine) * P + total / 2) / total);
    if (c1 <= c0) {  // no CTA of its own
        if (cta == (c0 < P ? c0 : P - 1)) *rb = rows;
        return;
    }
    if (cta < c0 || cta >= c1) return;
    const int64_t n = c1 - c0, l = cta - c0;
    *ra = l * rows / n;
    *rb = (l + 1) * rows / n;
}

// Byte offset of chunk j inside a row, and the shared-memory address of row
// `row`'s segment of the tile in a stage (it keeps the source's offset mod 16).
QDQ_DEV int64_t chunk_off(const DevDesc &d, int j) {
    return (int64_t)j * (kChunk / blk_weights(d.type)) * blk_bytes(d.type);
}
QDQ_DEV uint32_t seg_addr(const DevDesc &d, const Tile &t, uint32_t stage, int r) {
    if (t.whole) return stage + (uint32_t)((uintptr_t)(d.W + t.row0 * d.rb) & 15) + (uint32_t)r * d.rb;
    const uint8_t *src = d.W + (t.row0 + r) * d.rb + chunk_off(d, t.chunk);
    return stage + (uint32_t)r * seg_pitch(seg_bytes(d, t.ccols)) + (uint32_t)((uintptr_t)src & 15);
}
// Producer side: bulk copies of the tile into a stage (see copy_span).
QDQ_DEV uint32_t tile_copy(const DevDesc &d, const Tile &t, uint32_t stage, uint32_t bar, int mode) {
    const uint8_t *w_end = d.W + d.rows * (int64_t)d.rb;
    if (t.whole) return copy_span(d.W + t.row0 * d.rb, (uint32_t)t.nrows * d.rb, w_end, stage, bar, mode);
    const int seg = seg_bytes(d, t.ccols), pitch = seg_pitch(seg);
    const int64_t off = chunk_off(d, t.chunk);
    uint32_t total = 0;
    for (int r = 0; r < t.nrows; ++r)
        total += copy_span(d.W + (t.row0 + r) * d.rb + off, (uint32_t)seg, w_end, stage + (uint32_t)(r * pitch), bar,
                           mode);
    return total;
}

// ---------------------------------------------------------------------------
// x slices in a warp's area. A slice is 256 floats in 64 16-byte units; unit
// u = 16 q + i (lane quarter q reads units 16 q .. 16 q + 15) is stored at
// 16 q + (i ^ 2 q), so the four quarters of a warp read four bank groups.
// ---------------------------------------------------------------------------
QDQ_DEV int xunit(int u) { return (u & ~15) | ((u & 15) ^ ((u >> 3) & 6)); }

// Stages x[col0 .. col0 + 2048 * (w1 - w0)) for warp w: slices of chunks w0..w1-1
// in every copy kind, and the sub-block sums when Q4_K reads this x.
QDQ_DEV void stage_x(const DevDesc &d, int w0, int w1, int w, int lane, float *area) {
    const int kinds = d.kinds, nk = nkinds(kinds);
    const int sums_off = (w1 - w0) * kSlice * nk;
    constexpr int kMaxWin = kXFloats / kSlice;
    float4 v[2 * kMaxWin];
#pragma unroll
    for (int j = 0; j < kMaxWin; ++j) {
        const int col = (w0 + j) * kChunk + w * kSlice + 8 * lane;
        const bool ok = (w0 + j) < w1 && col < d.cols;
        v[2 * j] = ok ? __ldcg((const float4 *)(d.x + col)) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[2 * j + 1] = ok ? __ldcg((const float4 *)(d.x + col + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int u0 = xunit(2 * lane), u1 = xunit(2 * lane + 1);
#pragma unroll
    for (int j = 0; j < kMaxWin; ++j) {
        if (w0 + j >= w1) break;
        float *base = area + j * kSlice * nk;
        int slot = 0;
        if (kinds & 1) {  // plain
            ((float4 *)(base + slot * kSlice))[u0] = v[2 * j];
            ((float4 *)(base + slot * kSlice))[u1] = v[2 * j + 1];
            ++slot;
        }
        if (kinds & 2) {  // Q4_K: columns 0..31 of each 64 meet low nibbles
            const bool hi = (lane & 7) >= 4;
            const float4 a = v[2 * j], b = v[2 * j + 1];
            ((float4 *)(base + slot * kSlice))[u0] =
                make_float4(a.x * nibble_scale(hi, 0), a.y * nibble_scale(hi, 1), a.z * nibble_scale(hi, 2),
                            a.w * nibble_scale(hi, 3));
            ((float4 *)(base + slot * kSlice))[u1] =
                make_float4(b.x * nibble_scale(hi, 0), b.y * nibble_scale(hi, 1), b.z * nibble_scale(hi, 2),
                            b.w * nibble_scale(hi, 3));
            ++slot;
            float s = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if ((lane & 3) == 0) area[sums_off + 8 * j + (lane >> 2)] = s;
        }
        if (kinds & 4) {  // q4_0: columns 0..15 of each 32 meet low nibbles
            const bool hi = (lane & 3) >= 2;
            const float4 a = v[2 * j], b = v[2 * j + 1];
            ((float4 *)(base + slot * kSlice))[u0] =
                make_float4(a.x * nibble_scale(hi, 0), a.y * nibble_scale(hi, 1), a.z * nibble_scale(hi, 2),
                            a.w * nibble_scale(hi, 3));
            ((float4 *)(base + slot * kSlice))[u1] =
                make_float4(b.x * nibble_scale(hi, 0), b.y * nibble_scale(hi, 1), b.z * nibble_scale(hi, 2),
                            b.w * nibble_scale(hi, 3));
        }
    }
    __syncwarp();
}

// The lane's 64 x values for its quarter c of the slice, as the units expect them:
// consecutive columns 64 c .. 64 c + 63 (Q4_K, q8_0, q4_0), or for Q6_K the four
// 16-column runs 128 h + 32 k + 16 m + (0..15), k = 0..3, with c = 2 h + m.
QDQ_DEV void load_xr(const float *slice, int type, int c, XSlice &xr) {
    const float4 *s4 = (const float4 *)slice;
    if (type == QDQ_Q6_K) {
        const int h = c >> 1, m = c & 1;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = s4[xunit(32 * h + 8 * k + 4 * m + i)];
                xr.v[8 * k + 2 * i] = bits2(__float_as_uint(v.x), __float_as_uint(v.y));
                xr.v[8 * k + 2 * i + 1] = bits2(__float_as_uint(v.z), __float_as_uint(v.w));
            }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 v = s4[xunit(16 * c + i)];
            xr.v[2 * i] = bits2(__float_as_uint(v.x), __float_as_uint(v.y));
            xr.v[2 * i + 1] = bits2(__float_as_uint(v.z), __float_as_uint(v.w));
        }
    }
}

// Rows r (and r + 8 when NR == 2) x the lane's 64 columns of the warp's slice.
// wrow[i] points at the slice in row i's segment; rows past the tile re-read the
// tile's last row and their results are dropped.
template <int NR>
QDQ_DEV void slice_dot(int type, const uint8_t *const *wrow, int c, int nblk, const XSlice &xr, float (&out)[NR]) {
    float acc[NR][1];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r][0] = 0.f;
    if (type == QDQ_Q4_K) unit_q4k<1, NR>(wrow, c, xr, nullptr, 0, 0, nullptr, 0, acc);
    else if (type == QDQ_Q6_K) unit_q6k<1, NR>(wrow, c, xr, nullptr, 0, 0, acc);
    else if (2 * c < nblk) {
        if (type == QDQ_Q8_0) unit_q8_0<1, NR>(wrow, c, nblk, xr, nullptr, 0, 0, acc);
        else unit_q4_0<1, NR>(wrow, c, nblk, xr, nullptr, 0, 0, acc);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) out[r] = acc[r][0];
}

// Shared-memory addresses of a tile's rows: whole rows are contiguous (one
// copy that keeps the source's offset mod 16); chunk segments sit at a fixed
// pitch, each keeping its own source offset mod 16.
struct RowGeo {
    uint32_t src_lo;  // low bits of the global address of row 0's first tile byte
    int rb;           // row bytes in global memory
    int pitch;        // stage pitch of chunk segments (0: whole rows)
};
QDQ_DEV const uint8_t *row_ptr(const uint8_t *stage_p, const RowGeo &g, int r) {
    if (g.pitch == 0) return stage_p + (g.src_lo & 15u) + (uint32_t)(r * g.rb);
    return stage_p + (uint32_t)(r * g.pitch) + ((g.src_lo + (uint32_t)(r * g.rb)) & 15u);
}

// This warp's slices of a tile, for one format: 256-column slices cw, cw + 8, ...
// of whole rows, or slice cw of a chunk. For each slice the x registers are
// loaded once and serve every pass of up to 16 rows; the warp's row partials go
// to its own column of the level buffer (stored for the first contribution,
// added otherwise).
template <int TYPE>
QDQ_DEV void tile_slices(const Tile &tl, const DevDesc &d, const uint8_t *stage_p, const RowGeo &geo,
                         const float *area, int cw, int r8, int c, float *mycol) {
    constexpr int QK = (TYPE == QDQ_Q4_K || TYPE == QDQ_Q6_K) ? 256 : 32;
    constexpr int SB = (kSlice / QK) * blk_bytes(TYPE);  // slice bytes
    constexpr int KIND = x_kind(TYPE);
    const int nk = nkinds(d.kinds);
    const int slot = __popc(d.kinds & ((1 << KIND) - 1));
    const int nslices = (tl.ccols + kSlice - 1) / kSlice;
    const int k0 = tl.whole ? cw : 8 * tl.chunk + cw;
    const int kend = tl.whole ? nslices : (cw < nslices ? k0 + 1 : k0);
    const int npass = (tl.nrows + kPassRows - 1) / kPassRows;
    bool fresh = tl.first;
    for (int k = k0; k < kend; k += kCW) {
        const int jw = (k >> 3) - tl.xw0;  // chunk of the slice in the x window
        XSlice xr;
        load_xr(area + jw * kSlice * nk + slot * kSlice, TYPE, c, xr);
        if constexpr (TYPE == QDQ_Q4_K) {
            const float *sums = area + tl.xwn * kSlice * nk + 8 * jw;
            xr.s0 = sums[2 * c];
            xr.s1 = sums[2 * c + 1];
        }
        const int kcols = d.cols - k * kSlice;
        const int nb = (kcols < kSlice ? kcols : kSlice) / QK;
        const uint32_t koff = (uint32_t)(tl.whole ? k : cw) * SB;
        for (int p = 0; p < npass; ++p) {
            const int rp = p * kPassRows, left = tl.nrows - rp;
            float o0 = 0.f, o1 = 0.f;
            if (left > 8) {
                const int rb = r8 + 8 < left ? rp + r8 + 8 : tl.nrows - 1;
                const uint8_t *wrow[2] = {row_ptr(stage_p, geo, rp + r8) + koff, row_ptr(stage_p, geo, rb) + koff};
                float acc[2][1] = {{0.f}, {0.f}};
                if constexpr (TYPE == QDQ_Q4_K) unit_q4k<1, 2>(wrow, c, xr, nullptr, 0, 0, nullptr, 0, acc);
                else if constexpr (TYPE == QDQ_Q6_K) unit_q6k<1, 2>(wrow, c, xr, nullptr, 0, 0, acc);
                else if (2 * c < nb) {
                    if constexpr (TYPE == QDQ_Q8_0) unit_q8_0<1, 2>(wrow, c, nb, xr, nullptr, 0, 0, acc);
                    else unit_q4_0<1, 2>(wrow, c, nb, xr, nullptr, 0, 0, acc);
                }
                o0 = acc[0][0];
                o1 = acc[1][0];
            } else {
                const int ra = r8 < left ? rp + r8 : tl.nrows - 1;
                const uint8_t *wrow[1] = {row_ptr(stage_p, geo, ra) + koff};
                float acc[1][1] = {{0.f}};
                if constexpr (TYPE == QDQ_Q4_K) unit_q4k<1, 1>(wrow, c, xr, nullptr, 0, 0, nullptr, 0, acc);
                else if constexpr (TYPE == QDQ_Q6_K) unit_q6k<1, 1>(wrow, c, xr, nullptr, 0, 0, acc);
                else if (2 * c < nb) {
                    if constexpr (TYPE == QDQ_Q8_0) unit_q8_0<1, 1>(wrow, c, nb, xr, nullptr, 0, 0, acc);
                    else unit_q4_0<1, 1>(wrow, c, nb, xr, nullptr, 0, 0, acc);
                }
                o0 = acc[0][0];
            }
            o0 += __shfl_xor_sync(0xffffffffu, o0, 1);
            o1 += __shfl_xor_sync(0xffffffffu, o1, 1);
            o0 += __shfl_xor_sync(0xffffffffu, o0, 2);
            o1 += __shfl_xor_sync(0xffffffffu, o1, 2);
            if (c == 0) {
                float *q = mycol + rp + r8;
                if (r8 < left) q[0] = fresh ? o0 : q[0] + o0;
                if (r8 + 8 < left) q[8] = fresh ? o1 : q[8] + o1;
            }
        }
        fresh = false;
    }
    if (fresh && c == 0)  // no slice of this warp in the tile: zero partials
        for (int rr = r8; rr < tl.nrows; rr += 8) mycol[rr] = 0.f;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int MAXD, int MAXL>
__global__ void __launch_bounds__(kThreads, 1) stream1_kernel(const __grid_constant__ StreamArgs<MAXD, MAXL> a) {
    using SM = Smem<MAXD>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *xareas = (float *)(smem + SM::kX);
    float *part = (float *)(smem + SM::kPart);
    uint64_t *dst = (uint64_t *)(smem + SM::kDst);
    int64_t *ranges = (int64_t *)(smem + SM::kRanges);
    const uint32_t ring_a = smem_u32(smem);
    const uint32_t full_a = smem_u32(smem + SM::kBars), empty_a = full_a + 8 * kSlots;
    // lvl: this CTA's consumers finished a level; dep: every CTA finished the
    // previous level (arrival by the control warp).
    const uint32_t lvl_a = empty_a + 8 * kSlots, dep_a = lvl_a + 8;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, P = gridDim.x;
    int *status = &s_status_s1;
    const bool levels_synced = a.counters != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(full_a + 8 * s, 1);
            mbar_init(empty_a + 8 * s, kCW);
        }
        mbar_init(lvl_a, kCW);
        mbar_init(dep_a, 1);
        fence_mbar_init();
    }
    for (int L = 0; L < a.nlevels; ++L)
        for (int g = a.level_start[L] + (int)threadIdx.x; g < a.level_start[L + 1]; g += kThreads)
            cta_rows_by_gemv(a, L, g, cta, P, &ranges[2 * g], &ranges[2 * g + 1]);
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        // A tile takes the next ring bytes; before copying, the producer waits (in
        // FIFO order) for the release of every live tile that overlaps them and of
        // the tile that last used the barrier slot.
        int t = 0, rel = 0;
        uint32_t next = 0;
        uint32_t *toff = (uint32_t *)(smem + SM::kRing), *tlen = toff + kSlots;
        walk(
            a, ranges, [](int) {},
            [&](const Tile &tl, int, const DevDesc &d) {
                const uint32_t bytes = tile_ring_bytes(d, tl.nrows, tl.whole, tl.ccols);
                const uint32_t o = ring_place(next, bytes);
                for (;;) {
                    bool block = rel < t && rel <= t - kSlots;
                    for (int j = rel; !block && j < t; ++j) {
                        const uint32_t jo = toff[j % kSlots], je = jo + tlen[j % kSlots];
                        block = o < je && jo < o + bytes;
                    }
                    if (!block) break;
                    mbar_wait(empty_a + 8 * (rel % kSlots), (rel / kSlots) & 1, status);
                    ++rel;
                }
                const int s = t % kSlots;
                toff[s] = o;
                tlen[s] = bytes;
                const uint32_t stage = ring_a + o, bar = full_a + 8 * s;
                const uint32_t nb = tile_copy(d, tl, stage, bar, kTail);
                mbar_arrive_expect_tx(bar, nb);  // releases the tail stores above
                tile_copy(d, tl, stage, bar, kBulk);
                ++t;
            },
            [](int) {});
        for (int i = t - kSlots > 0 ? t - kSlots : 0; i < t; ++i)  // no exit with copies in flight
            mbar_wait(full_a + 8 * (i % kSlots), (i / kSlots) & 1, status);
        return;
    }

    if (warp == 1) {
        // ------------------------------------------------------------ control
        // Publishes level L once this CTA's consumers have finished it, waits until
        // every CTA has, and releases the consumers into level L+1. lvl completes
        // one phase per level in which this CTA has tiles, and dep is arrived only
        // for such levels; neither can run two phases ahead of its waiter.
        if (!levels_synced) return;
        auto has_tiles = [&](int L) {
            for (int g = a.level_start[L]; g < a.level_start[L + 1]; ++g)
                if (ranges[2 * g] < ranges[2 * g + 1]) return true;
            return false;
        };
        int lvl_phase = 0;
        bool prev_had = has_tiles(0);
        for (int L = 1; L < a.nlevels; ++L) {
            if (lane == 0) S1_TR(L, 0);
            if (prev_had) mbar_wait_spin(lvl_a, (lvl_phase++) & 1, status);
            if (lane == 0) {
                S1_TR(L, 1);
                // The consumers' y stores are ordered before their arrivals (CTA
                // scope); the release makes them visible at GPU scope with the count.
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&a.counters[L - 1]) : "memory");
                wait_counter(&a.counters[L - 1], (unsigned)P, status, kWaitLimitNs);
                S1_TR(L, 2);
            }
            __syncwarp();
            const bool had = has_tiles(L);
            if (had && lane == 0) mbar_arrive(dep_a);
            prev_had = had;
        }
        if (prev_had) mbar_wait_spin(lvl_a, (lvl_phase++) & 1, status);
        if (lane == 0) {
            __threadfence();
            const unsigned old = atomicAdd(&a.counters[a.nlevels - 1], 1u);
            if (old == (unsigned)P - 1) {  // every CTA has passed every wait: reset for the next run
                for (int i = 0; i < a.nlevels; ++i) a.counters[i] = 0u;
                __threadfence();
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - kFirstCW;
    const int ctid = (int)threadIdx.x - 32 * kFirstCW;
    const int r8 = lane >> 2, c = lane & 3;
    float *area = xareas + cw * kXFloats;
    float *mypart = part + cw * kBufRows;
    int t = 0, cur_e = -1, cur_level = 0, tiles_in_level = 0, dep_phase = 0;
    int buf_rows = 0, rg_base = 0;
    uint32_t ring_next = 0;
    bool had_tiles = false, dep_pending = false;
    (void)cur_level;

    // Adds the eight warps' partials of every buffered row (warp order) and stores
    // y (adding to it for rows whose earlier columns were stored before).
    auto flush = [&]() {
        named_bar_sync(kFlushBar, kCW * 32);  // partials and addresses are in place
        for (int i = ctid; i < buf_rows; i += kCW * 32) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) sum += part[w * kBufRows + i];
            const uint64_t d = dst[i];
            float *yp = (float *)(uintptr_t)(d & ~(uint64_t)1);
            if (d & 1) sum += __ldcg(yp);
            *yp = sum;
        }
        named_bar_sync(kFlushBar, kCW * 32);  // the buffer may be refilled
        buf_rows = 0;
    };

    walk(
        a, ranges,
        [&](int L) {
            cur_level = L;
            tiles_in_level = 0;
            dep_pending = L > 0 && levels_synced;
        },
        [&](const Tile &tl, int e, const DevDesc &d) {
            had_tiles = true;
            if (cw == 0 && lane == 0 && tiles_in_level == 0) S1_TR(cur_level, 4);
            if (e != cur_e) {
                if (dep_pending) {  // the previous level is complete on every CTA
                    mbar_wait_spin(dep_a, (dep_phase++) & 1, status);
                    dep_pending = false;
                }
                cur_e = e;
                stage_x(d, tl.xw0, tl.xw0 + tl.xwn, cw, lane, area);
            }
            if (tl.first) {  // a new row group: its rows in the partial buffer
                // Rows whose earlier columns sit in this buffer are stored first.
                if (buf_rows + tl.nrows > kBufRows || (!tl.first_win && buf_rows > 0)) flush();
                rg_base = buf_rows;
                buf_rows += tl.nrows;
                if (cw == 0)
                    for (int i = lane; i < tl.nrows; i += 32)
                        dst[rg_base + i] = (uint64_t)(uintptr_t)(d.y + tl.row0 + i) | (tl.first_win ? 0u : 1u);
            }
            if (cw == 0 && lane == 0 && tiles_in_level == 0) S1_TR(cur_level, 5);
            if (cw == 0 && lane == 0 && tiles_in_level < 7) S1_TRC(cur_level, 8 + 3 * tiles_in_level);
            const uint32_t toffs = ring_place(ring_next, tile_ring_bytes(d, tl.nrows, tl.whole, tl.ccols));
            const int s = t % kSlots;
            mbar_wait(full_a + 8 * s, (t / kSlots) & 1, status);
            if (cw == 0 && lane == 0 && tiles_in_level == 0) S1_TR(cur_level, 6);
            if (cw == 0 && lane == 0 && tiles_in_level < 7) S1_TRC(cur_level, 9 + 3 * tiles_in_level);
            ++tiles_in_level;

            {
                const uint8_t *stage_p = smem + toffs;
                RowGeo geo;
                geo.rb = d.rb;
                if (tl.whole) {
                    geo.src_lo = (uint32_t)(uintptr_t)(d.W + tl.row0 * d.rb);
                    geo.pitch = 0;
                } else {
                    geo.src_lo = (uint32_t)(uintptr_t)(d.W + tl.row0 * d.rb + chunk_off(d, tl.chunk));
                    geo.pitch = seg_pitch(seg_bytes(d, tl.ccols));
                }
                float *mycol = mypart + rg_base;
                switch (d.type) {
                    case QDQ_Q4_K: tile_slices<QDQ_Q4_K>(tl, d, stage_p, geo, area, cw, r8, c, mycol); break;
                    case QDQ_Q6_K: tile_slices<QDQ_Q6_K>(tl, d, stage_p, geo, area, cw, r8, c, mycol); break;
                    case QDQ_Q8_0: tile_slices<QDQ_Q8_0>(tl, d, stage_p, geo, area, cw, r8, c, mycol); break;
                    default: tile_slices<QDQ_Q4_0>(tl, d, stage_p, geo, area, cw, r8, c, mycol); break;
                }
            }
            __syncwarp();
            if (cw == 0 && lane == 0 && tiles_in_level <= 7) S1_TRC(cur_level, 7 + 3 * tiles_in_level);
            if (lane == 0) mbar_arrive(empty_a + 8 * s);
            ++t;
        },
        [&](int) {
            if (buf_rows > 0) flush();
            if (cw == 0 && lane == 0) S1_TR(cur_level, 7);
            if (levels_synced && had_tiles) {
                __syncwarp();
                if (lane == 0) mbar_arrive(lvl_a);  // release (CTA scope) of the level's y stores
            }
            had_tiles = false;
            dep_pending = false;  // a level without tiles here needs no release
        });
}

}  // namespace s1

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int MAXD, int MAXL>
static int launch1(const void *args, int grid, bool cooperative, cudaStream_t stream) {
    auto kern = s1::stream1_kernel<MAXD, MAXL>;
    constexpr int smem = s1::Smem<MAXD>::kBytes;
    RelaxedCaptureScope relaxed;  // the first launch sets the kernel's attributes
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 63]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
            cudaGetLastError();
            return QDQ_ERR_CUDA;
        }
        attr_done[dev & 63] = true;
    }
    void *params[] = {const_cast<void *>(args)};
    const cudaError_t e =
        cooperative
            ? cudaLaunchCooperativeKernel((const void *)kern, dim3(grid), dim3(s1::kThreads), params, (size_t)smem,
                                          stream)
            : cudaLaunchKernel((const void *)kern, dim3(grid), dim3(s1::kThreads), params, (size_t)smem, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
}

int stream1_launch(const void *args, bool big, bool cooperative, int grid, cudaStream_t stream) {
    return big ? launch1<kMaxPlanDescs, kMaxPlanLevels>(args, grid, cooperative, stream)
               : launch1<kMaxGroupDescs, 1>(args, grid, cooperative, stream);
}

int take_status_stream1() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, s_status_s1, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(s_status_s1, &zero, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    return v;
}

}  // namespace qdq
