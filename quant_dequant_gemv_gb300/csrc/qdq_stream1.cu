// qdq_stream1.cu -- fused dequant-GEMV on CUDA cores for small batches (batch
// widths 1, 2, 4, 8): single GEMVs, groups and multi-level plans such as a decode
// step.
//
// "S21 The Capstone: picoLM, in Python", section 3 (fused dequant + dot: only the
// quantised bytes cross the memory bus, decoded in registers into the dot
// product) and section 4 (the per-layer projections of a decode step, each level
// waiting for the previous one); "PETIT" (gemv_q8 / gemv_q4, rows of 32-weight
// blocks, weights stored out x in).
//
// One persistent CTA per SM, warp-specialised, with the reduction dimension
// split across the consumer warps:
//  * Tiles. A whole-row tile holds up to 64 complete rows; rows too long for
//    eight per tile, or whose x does not fit the x window, are cut into
//    2048-column chunks of up to 32 rows. Work is split by 256-column slices
//    (one Q4_K / Q6_K super-block, eight q8_0 / q4_0 blocks): lane 4 r + c
//    covers row r (and r + 8) and quarter c of a slice, 64 weights per row.
//    At batch width 1 fifteen consumer warps take the tile's (row pass, slice)
//    units in turn, with passes of 8 or 16 rows, so a level with a dozen rows
//    per CTA still gives every warp a unit. At widths 2-8 eight consumer warps
//    each own the slices w, w + 8, ... of every row.
//  * x. The consumer warps stage the window's x (plain and/or pre-scaled
//    copies, every batch column) into one CTA-wide buffer and read it inside
//    the word loop; the loads of a warp touch at most four 16-byte units each,
//    which shared memory serves as broadcasts.
//  * Partials. A warp keeps its row partials for the whole level in a
//    shared-memory buffer (the chunks of a row add up in place); at the end of
//    the level (or when the buffer is full) the consumer warps meet once, add
//    the warps' partials of each row in warp order and store y.
//  * Warp 0 streams tiles HBM -> shared memory with 1-D bulk copies into a byte
//    ring and fetches ahead across level boundaries (W does not depend on x).
//    The consumers own the level dependency: one device-wide counter per level,
//    raised by one consumer thread after the level's y stores and polled by it
//    before the next level's x is read (the other consumer warps wait at a
//    named barrier).
//  * Every wait is bounded (qdq_device.cuh).
#include <cstdio>
#include <type_traits>

#include <cuda_fp16.h>

#include "qdq_stream_common.cuh"

namespace qdq {

static __device__ int s_status_s1;

// Phase timestamps for performance analysis, compiled in only with -DQDQ_TRACE:
// trace[(cta * nlevels + level) * 32 + slot] = %globaltimer (S1_TR) or the SM's
// clock64 (S1_TRC, per-tile phases of the first consumer warp). Slots: 1-2 level
// dependency wait, 3 units done, 4-7 consumer level phases, 8-28 per tile (before the full wait, after it,
// after processing), 29 producer reaches the level's first tile, 30-31 producer
// has issued the level's first and second tile.
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

constexpr int kFirstCW = 1;                       // warp 0 producer, then the consumers
constexpr int kTileRows = 64;                     // rows of a whole-row tile
constexpr int kChunkRows = 32;                    // rows of a chunked tile
constexpr int kChunk = 2048;                      // columns of a chunk: kSlicesPerChunk slices of kSlice
constexpr int kSlice = 256;
constexpr int kSlicesPerChunk = kChunk / kSlice;
constexpr int kSlots = 8;                         // full/empty barrier pairs (tiles in the ring)
constexpr int kFlushBar = 1;                      // named barrier of the consumer warps
constexpr int kDepBar = 2;                        // the consumer warps wait here for a level dependency
constexpr int kPartFloats = 6144;                 // level partial buffer: [warp][row][batch column]

// Per batch width BT (1, 2, 4, 8). x for every batch column of the staged window
// sits in one CTA-wide buffer and is read inside the word loop. Batch 1 runs
// fifteen consumer warps that take (row pass, slice) work units in turn; wider
// batches run eight, warp w owning slices w, w + 8, ... of every tile.
template <int BT>
struct Cfg {
    // consumer warps; at batch 1 the producer and fifteen consumers make sixteen
    // warps, four per scheduler, whose registers (up to 128 each) fill the file
    static constexpr int kCW = BT == 1 ? 15 : 8;
    static constexpr int kThreads = 32 * (kCW + kFirstCW);
    static constexpr int kRingBytes = BT == 1 ? 153600 : 114688;   // W ring: tiles packed in order
    static constexpr int kMaxTileBytes = kRingBytes / 2;           // at least two tiles in flight
    static constexpr int kXFloats = BT == 1 ? 10240 : 20480;       // x staging (CTA-wide)
    // rows of the level partial buffer (a multiple of 8 keeps every later region aligned)
    static constexpr int kBufRows = (kPartFloats / (kCW * BT)) & ~7;
    static constexpr int kNR = BT <= 4 ? 2 : 1;                    // rows per lane in one pass (BT > 1)
};

// Shared memory layout (bytes). The ring starts at 0 (1024-aligned base).
template <int BT, int MAXD>
struct Smem {
    static constexpr int kX = Cfg<BT>::kRingBytes;
    static constexpr int kPart = kX + Cfg<BT>::kXFloats * 4;
    static constexpr int kDst = kPart + kPartFloats * 4;               // y address of each buffer row
    static constexpr int kDstStride = kDst + Cfg<BT>::kBufRows * 8;    // its batch-column stride (BT > 1) or scale (BT = 1)
    static constexpr int kRanges = kDstStride + Cfg<BT>::kBufRows * 4;
    static constexpr int kRing = kRanges + 2 * MAXD * 8;              // producer: live tiles' ring ranges
    static constexpr int kBars = kRing + 2 * kSlots * 4;
    static constexpr int kRed = kBars + (2 * kSlots + 2) * 8;          // per-warp partial sums of x^2 [warp][b]
    static constexpr int kBytes = kRed + 16 * 8 * 4;
};
template <int BT, int MAXD>
constexpr bool smem_aligned() {
    using S = Smem<BT, MAXD>;
    return S::kX % 16 == 0 && S::kPart % 16 == 0 && S::kDst % 8 == 0 && S::kRanges % 8 == 0 && S::kRing % 4 == 0 &&
           S::kBars % 8 == 0;
}
static_assert(smem_aligned<1, kMaxPlanDescs>() && smem_aligned<1, kMaxGroupDescs>() &&
                  smem_aligned<2, kMaxPlanDescs>() && smem_aligned<2, kMaxGroupDescs>() &&
                  smem_aligned<4, kMaxPlanDescs>() && smem_aligned<4, kMaxGroupDescs>() &&
                  smem_aligned<8, kMaxPlanDescs>() && smem_aligned<8, kMaxGroupDescs>(),
              "every shared-memory region at its access alignment (float4 x, int64 ranges, mbarriers)");
static_assert(Smem<1, kMaxPlanDescs>::kBytes <= 227 * 1024, "shared memory budget");
static_assert(Smem<2, kMaxPlanDescs>::kBytes <= 227 * 1024, "shared memory budget");
static_assert(Smem<8, kMaxPlanDescs>::kBytes <= 227 * 1024, "shared memory budget");

// ---------------------------------------------------------------------------
// Tiles: identical sequence for the producer and the consumers.
// A whole-row tile holds up to 64 complete rows and every chunk of their x. It
// is one contiguous bulk copy, except for rows whose length is a multiple of 128
// bytes read with 32-bit loads: those are copied row by row to a pitch 16 bytes
// longer, so that the eight rows a warp reads at once fall in different shared-
// memory banks. Rows too long for 8 per stage are cut into 2048-column chunks of
// up to 32 rows, copied row segment by row segment at a padded pitch.
// ---------------------------------------------------------------------------
struct Tile {
    int g;            // GEMV (desc index)
    int nrows;        // 1..64 (whole rows) or 1..32 (chunked)
    int64_t row0;
    int chunk;        // chunked: the 2048-column chunk; whole rows: 0
    int ccols;        // columns of the tile (whole rows: all of them)
    int xw0;          // first chunk of the staged x window (chunk - xw0 indexes it)
    int xwn;          // chunks in that window
    bool whole;       // complete rows, contiguous in the stage
    bool first;       // first chunk of this row group in the window
    bool last;        // last chunk of this row group in the window
    bool first_win;   // the window starts at column 0 (y is stored, not accumulated)
    bool attn;        // attention heads row0 .. row0 + nrows - 1 (no weights, no ring slot)
    int skinds;       // x copy kinds staged for this tile's epoch
};

QDQ_DEV int nkinds(int kinds) { return __popc(kinds & 7); }
// x floats staged per chunk (CTA-wide): the chunk's 2048 columns of every batch
// column in every kind.
template <int BT>
QDQ_DEV int xfloats_per_chunk(int kinds) {
    return kChunk * nkinds(kinds) * BT;
}
template <int BT>
QDQ_DEV int window_chunks(int kinds) {
    const int w = Cfg<BT>::kXFloats / xfloats_per_chunk<BT>(kinds);
    return w < 1 ? 1 : w;
}
// The kinds staged for a GEMV: every kind its level reads from this x when one
// chunk of them fits, else only its own (the level's GEMVs then stage in turn).
template <int BT>
QDQ_DEV int staged_kinds(const DevDesc &d) {
    return xfloats_per_chunk<BT>(d.kinds) <= Cfg<BT>::kXFloats ? d.kinds : 1 << x_kind(d.type);
}
// Bytes of one row segment of a chunk, and the stage pitch of such segments.
QDQ_DEV int seg_bytes(const DevDesc &d, int ccols) { return (ccols / blk_weights(d.type)) * blk_bytes(d.type); }
QDQ_DEV int seg_pitch(int seg) { return ((seg + 15) & ~15) + 16; }
// Whole rows copied one by one to a padded pitch (see the tile comment above):
// the formats read with 32-bit loads (Q6_K, q8_0, q4_0), rows of at least 2 KiB
// whose length is a multiple of 128 bytes, and a 16-byte aligned matrix.
QDQ_DEV bool rows_padded(const DevDesc &d) {
    return d.type != QDQ_Q4_K && d.rb >= 2048 && (d.rb & 127) == 0 && ((uintptr_t)d.W & 15) == 0;
}
QDQ_DEV int whole_pitch(const DevDesc &d) { return rows_padded(d) ? d.rb + 16 : d.rb; }
// Rows of a whole-row tile (a multiple of 8 up to 64), or 0 when fewer than 8
// rows fit a stage or the row's x does not fit one window.
template <int BT>
QDQ_DEV int whole_rows(const DevDesc &d, int skinds) {
    const int nch = (d.cols + kChunk - 1) / kChunk;
    const int cap = (Cfg<BT>::kMaxTileBytes - 32) / whole_pitch(d);
    if (cap < 8 || nch > window_chunks<BT>(skinds)) return 0;
    constexpr int rmax = kTileRows < Cfg<BT>::kBufRows ? kTileRows : Cfg<BT>::kBufRows;  // fits the partial buffer
    return cap >= rmax ? rmax : cap & ~7;
}
template <int BT>
QDQ_DEV int chunk_rows(const DevDesc &d) {
    const int cap = Cfg<BT>::kMaxTileBytes / seg_pitch(seg_bytes(d, kChunk));
    return cap < kChunkRows ? (cap < 1 ? 1 : cap) : kChunkRows;
}

// Bytes a tile takes in the ring (copy_span may start up to 15 bytes before and
// end up to 15 bytes after the tile's rows; padded rows and chunk segments sit at
// their pitch).
QDQ_DEV uint32_t tile_ring_bytes(const DevDesc &d, int nrows, bool whole, int ccols) {
    const uint32_t b = whole ? (uint32_t)(nrows * whole_pitch(d) + 32) : (uint32_t)(nrows * seg_pitch(seg_bytes(d, ccols)));
    return (b + 127u) & ~127u;
}
// Next tile's offset in the ring: packed after the previous one, or at 0 when it
// would not fit before the end. Producer and consumers run the same sequence.
template <int BT>
QDQ_DEV uint32_t ring_place(uint32_t &next, uint32_t bytes) {
    if (next + bytes > (uint32_t)Cfg<BT>::kRingBytes) next = 0;
    const uint32_t o = next;
    next += bytes;
    return o;
}

// on_begin(L) / on_end(L) around each level; on_tile(tile, epoch, desc) for every
// tile. An epoch is one staged x window: (level, x, columns, window).
template <int BT, bool ATTN, class A, class FBegin, class FTile, class FEnd>
QDQ_DEV void walk(const A &a, const int64_t *ranges, FBegin &&on_begin, FTile &&on_tile, FEnd &&on_end) {
    int epoch = -1;
    for (int L = 0; L < a.nlevels; ++L) {
        on_begin(L);
        const float *ex = nullptr;
        int ew = -1, ecols = -1, ekinds = -1;
        for (int g = a.level_start[L]; g < a.level_start[L + 1]; ++g) {
            const int64_t ra = ranges[2 * g], rb = ranges[2 * g + 1];
            if (ra >= rb) continue;
            const DevDesc d = a.d[g];
            if (ATTN && d.type == kTypeAttn) {
                Tile t{};
                t.g = g;
                t.row0 = ra;
                t.nrows = (int)(rb - ra);
                t.attn = true;
                on_tile(t, epoch, d);
                continue;
            }
            const int nch = (d.cols + kChunk - 1) / kChunk;
            const int n = (int)(rb - ra);  // rows of one GEMV on one CTA
            const int sk = staged_kinds<BT>(d);
            const int wr = whole_rows<BT>(d, sk);
            if (wr > 0) {
                if (d.x != ex || 0 != ew || d.cols != ecols || sk != ekinds) {
                    ++epoch;
                    ex = d.x;
                    ew = 0;
                    ecols = d.cols;
                    ekinds = sk;
                }
                for (int r = 0; r < n; r += wr) {
                    Tile t{};
                    t.g = g;
                    t.nrows = n - r < wr ? n - r : wr;
                    t.row0 = ra + r;
                    t.chunk = 0;
                    t.ccols = d.cols;
                    t.xw0 = 0;
                    t.xwn = nch;
                    t.whole = true;
                    t.first = t.last = t.first_win = true;
                    t.skinds = sk;
                    on_tile(t, epoch, d);
                }
                continue;
            }
            const int wmax = window_chunks<BT>(sk);
            const int nrmax = chunk_rows<BT>(d);
            const int ntg = (n + nrmax - 1) / nrmax;
            const int nbase = n / ntg, nextra = n - nbase * ntg;
            for (int w0 = 0; w0 < nch; w0 += wmax) {
                const int w1 = nch < w0 + wmax ? nch : w0 + wmax;
                if (d.x != ex || w0 != ew || d.cols != ecols || sk != ekinds) {
                    ++epoch;
                    ex = d.x;
                    ew = w0;
                    ecols = d.cols;
                    ekinds = sk;
                }
                int64_t r = ra;
                for (int tg = 0; tg < ntg; ++tg) {
                    const int nr = nbase + (tg < nextra ? 1 : 0);
                    for (int j = w0; j < w1; ++j) {
                        Tile t{};
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
                        t.skinds = sk;
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
template <bool ATTN, class A>
QDQ_DEV void cta_rows_by_gemv(const A &a, int L, int g, int cta, int P, int64_t *ra, int64_t *rb) {
    if (ATTN && a.d[g].type == kTypeAttn) {  // an attention level (alone in its level): heads over the CTAs
        const int64_t heads = a.d[g].rows, n = heads < P ? heads : P;
        *ra = *rb = 0;
        if (cta < n) {
            *ra = cta * heads / n;
            *rb = (cta + 1) * heads / n;
        }
        return;
    }
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

// Byte offset of chunk j inside a row.
QDQ_DEV int64_t chunk_off(const DevDesc &d, int j) {
    return (int64_t)j * (kChunk / blk_weights(d.type)) * blk_bytes(d.type);
}
// n copies of len bytes, src advancing by sstride and dst by dstride: every
// address and length a multiple of 16, so nothing is over-read.
QDQ_DEV void copy_rows(const uint8_t *src, int64_t sstride, uint32_t dst, uint32_t dstride, uint32_t len, int n,
                       uint32_t bar) {
    const uint64_t pol = policy_evict_first();
    for (int r = 0; r < n; ++r, src += sstride, dst += dstride) bulk_g2s_hint(dst, src, len, bar, pol);
}
// Producer side: bulk copies of the tile into a stage. Returns the bulk byte
// count; mode kTail stores the trailing bytes of an unaligned matrix end, kBulk
// issues the copies (see copy_span).
QDQ_DEV uint32_t tile_copy(const DevDesc &d, const Tile &t, uint32_t stage, uint32_t bar, int mode) {
    const uint8_t *w_end = d.W + d.rows * (int64_t)d.rb;
    if (t.whole) {
        if (!rows_padded(d)) return copy_span(d.W + t.row0 * d.rb, (uint32_t)t.nrows * d.rb, w_end, stage, bar, mode);
        if (mode & kBulk) copy_rows(d.W + t.row0 * d.rb, d.rb, stage, (uint32_t)whole_pitch(d), (uint32_t)d.rb, t.nrows, bar);
        return (uint32_t)(t.nrows * d.rb);
    }
    const int seg = seg_bytes(d, t.ccols), pitch = seg_pitch(seg);
    const int64_t off = chunk_off(d, t.chunk);
    const uint8_t *src = d.W + t.row0 * d.rb + off;
    if ((((uintptr_t)src | (uintptr_t)d.rb | (uintptr_t)seg) & 15) == 0) {  // every segment aligned
        if (mode & kBulk) copy_rows(src, d.rb, stage, (uint32_t)pitch, (uint32_t)seg, t.nrows, bar);
        return (uint32_t)(t.nrows * seg);
    }
    uint32_t total = 0;
    for (int r = 0; r < t.nrows; ++r)
        total += copy_span(d.W + (t.row0 + r) * d.rb + off, (uint32_t)seg, w_end, stage + (uint32_t)(r * pitch), bar,
                           mode);
    return total;
}

// ---------------------------------------------------------------------------
// x in shared memory. A 256-float slice is 64 16-byte units; unit u = 16 q + i
// (lane quarter q reads units 16 q .. 16 q + 15) is stored at 16 q + (i ^ 2 q),
// so the four quarters of a warp read four bank groups.
// ---------------------------------------------------------------------------
QDQ_DEV int xunit(int u) { return (u & ~15) | ((u & 15) ^ ((u >> 3) & 6)); }

// ---------------------------------------------------------------------------
// x for every batch column sits in one CTA-wide buffer: per chunk of the window
// (stride xfloats_per_chunk<BT>), kind slot k, column b and slice w at
// (k * BT + b) * 2048 + w * 256 (swizzled units). The consumer warps stage
// (chunk, slice) pairs in turn: warp cw takes pairs cw, cw + ncw, ...
// ---------------------------------------------------------------------------
// rmsnorm of the GEMV input ("S21 The Capstone: picoLM, in Python", section 4:
// rmsnorm(xb, x, weight, dim) before the q/k/v and gate/up projections): inv[b] =
// 1 / sqrt(mean over the cols entries of x_b^2 + eps) for each batch column. The
// consumer warps sum strided float4 of the whole of x (not only the staged
// window), then every thread adds the warps' sums in warp order, so every
// thread holds the same inv.
template <int BT>
QDQ_DEV void rms_scale(const DevDesc &d, const DescEx &ex, int batch, int cw, int ncw, int lane, float *red,
                       float (&inv)[BT]) {
    float ss[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) ss[b] = 0.f;
    for (int c = 4 * (cw * 32 + lane); c < d.cols; c += 4 * 32 * ncw) {
#pragma unroll
        for (int b = 0; b < BT; ++b)
            if (b < batch) {
                const float4 v = __ldcg((const float4 *)(d.x + (int64_t)b * d.cols + c));
                ss[b] += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
            }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss[b] += __shfl_xor_sync(0xFFFFFFFFu, ss[b], o);
        if (lane == 0) red[cw * 8 + b] = ss[b];
    }
    named_bar_sync(kFlushBar, ncw * 32);
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float t = 0.f;
        for (int w = 0; w < ncw; ++w) t += red[w * 8 + b];
        inv[b] = 1.0f / sqrtf(t / (float)d.cols + ex.eps);
    }
}

QDQ_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

// The raw values behind x[b][col..col+7]: x itself and the operand of its option
// (the rmsnorm weight or, for SwiGLU, the up projection; x holds the gate), all
// four loads issued together (one round trip to L2 for the slice, not one per
// operand).
struct XRaw {
    float4 a, c, pa, pc;
};

QDQ_DEV XRaw x_load(const DevDesc &d, const DescEx &ex, int b, int col, bool ok) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    XRaw r{z, z, z, z};
    if (!ok) return r;
    const float *xr = d.x + (int64_t)b * d.cols + col;
    const int xop = desc_xop(d);
    if (xop == QDQ_X_SWIGLU || xop == QDQ_X_MUL) {
        const float *ur = ex.x2 + (int64_t)b * d.cols + col;
        r.a = __ldcg((const float4 *)xr);
        r.c = __ldcg((const float4 *)(xr + 4));
        r.pa = __ldcg((const float4 *)ur);
        r.pc = __ldcg((const float4 *)(ur + 4));
    } else if (xop == QDQ_X_RMSNORM) {
        r.a = __ldcg((const float4 *)xr);
        r.c = __ldcg((const float4 *)(xr + 4));
        r.pa = __ldg((const float4 *)(ex.nw + col));
        r.pc = __ldg((const float4 *)(ex.nw + col + 4));
    } else {
        r.a = __ldcg((const float4 *)xr);
        r.c = __ldcg((const float4 *)(xr + 4));
    }
    return r;
}

// The value the dot product reads (QDQ_X_*): as stored, rmsnorm-scaled by s,
// silu(gate) * up, or x * x2.
QDQ_DEV float4 x_apply(int xop, float s, float4 v, float4 p) {
    if (xop == QDQ_X_RMSNORM) return make_float4(v.x * s * p.x, v.y * s * p.y, v.z * s * p.z, v.w * s * p.w);
    if (xop == QDQ_X_SWIGLU)
        return make_float4(silu(v.x) * p.x, silu(v.y) * p.y, silu(v.z) * p.z, silu(v.w) * p.w);
    if (xop == QDQ_X_MUL) return make_float4(v.x * p.x, v.y * p.y, v.z * p.z, v.w * p.w);
    return v;
}

// The value the dot product reads at x[b][col..col+3] (QDQ_X_*): as stored,
// rmsnorm-scaled, or silu(gate) * up.
template <int BT>
QDQ_DEV float4 x_in(const DevDesc &d, const DescEx &ex, int b, int col, int off, const float (&inv)[BT], float4 v) {
    const int xop = desc_xop(d);
    if (xop == QDQ_X_RMSNORM) {
        const float4 w = __ldg((const float4 *)(ex.nw + col + off));
        const float s = inv[b];
        return make_float4(v.x * s * w.x, v.y * s * w.y, v.z * s * w.z, v.w * s * w.w);
    }
    if (xop == QDQ_X_SWIGLU) {
        const float4 u = __ldcg((const float4 *)(ex.x2 + (int64_t)b * d.cols + col + off));
        return make_float4(silu(v.x) * u.x, silu(v.y) * u.y, silu(v.z) * u.z, silu(v.w) * u.w);
    }
    return v;
}

// FUSED_LOADS (the model's instantiation): x and its option operand loaded
// together (x_load), QDQ_X_MUL included; otherwise (no QDQ_X_MUL there) the
// operand is loaded where it is applied, which keeps the GEMV-only
// instantiations within their registers.
template <int BT, bool FUSED_LOADS = false>
QDQ_DEV void stage_xb(const DevDesc &d, const DescEx &ex, int kinds, int batch, int w0, int w1, int cw, int ncw,
                      int lane, const float (&inv)[BT], float *xbuf, float *sumsq = nullptr) {
    const int stride = xfloats_per_chunk<BT>(kinds);
    const int u0 = xunit(2 * lane), u1 = xunit(2 * lane + 1);
    const int xop = desc_xop(d);
    for (int i = cw; i < (w1 - w0) * kSlicesPerChunk; i += ncw) {
        const int j = i / kSlicesPerChunk, w = i % kSlicesPerChunk;
        float *chunk = xbuf + j * stride;
        const int col = (w0 + j) * kChunk + w * kSlice + 8 * lane;
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            const bool ok = b < batch && col < d.cols;
            float4 ra, rc, a, c;
            if constexpr (FUSED_LOADS) {
                const XRaw r = x_load(d, ex, b, col, ok);
                ra = r.a;
                rc = r.c;
                a = ok ? x_apply(xop, inv[b], ra, r.pa) : ra;
                c = ok ? x_apply(xop, inv[b], rc, r.pc) : rc;
            } else {
                const float *xr = d.x + (int64_t)b * d.cols + col;
                ra = ok ? __ldcg((const float4 *)xr) : make_float4(0.f, 0.f, 0.f, 0.f);
                rc = ok ? __ldcg((const float4 *)(xr + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
                a = ok ? x_in<BT>(d, ex, b, col, 0, inv, ra) : ra;
                c = ok ? x_in<BT>(d, ex, b, col, 4, inv, rc) : rc;
            }
            if (sumsq != nullptr && b == 0)  // this lane's share of sum x^2 (rmsnorm folded into the flush)
                *sumsq += ((ra.x * ra.x + ra.y * ra.y) + (ra.z * ra.z + ra.w * ra.w)) +
                          ((rc.x * rc.x + rc.y * rc.y) + (rc.z * rc.z + rc.w * rc.w));
            int slot = 0;
            if (kinds & 1) {
                float4 *sl = (float4 *)(chunk + (slot * BT + b) * kChunk + w * kSlice);
                sl[u0] = a;
                sl[u1] = c;
                ++slot;
            }
            if (kinds & 4) {  // q4_0: columns 0..15 of each 32 meet low nibbles
                const bool hi = (lane & 3) >= 2;
                float4 *sl = (float4 *)(chunk + (slot * BT + b) * kChunk + w * kSlice);
                sl[u0] = make_float4(a.x * nibble_scale(hi, 0), a.y * nibble_scale(hi, 1), a.z * nibble_scale(hi, 2),
                                     a.w * nibble_scale(hi, 3));
                sl[u1] = make_float4(c.x * nibble_scale(hi, 0), c.y * nibble_scale(hi, 1), c.z * nibble_scale(hi, 2),
                                     c.w * nibble_scale(hi, 3));
            }
        }
    }
}

// x pair units of column b: xs points at column 0's slice; columns are 2048 apart.
QDQ_DEV void xpairs_b(const float *xs, int b, int u, uint64_t &p0, uint64_t &p1) {
    const float4 v = ((const float4 *)(xs + b * kChunk))[xunit(u)];
    p0 = bits2(__float_as_uint(v.x), __float_as_uint(v.y));
    p1 = bits2(__float_as_uint(v.z), __float_as_uint(v.w));
}

// Q4_K, NR rows x BT columns: each word is decoded once, into exact weights, and
// every weight meets every column. Lane quarter c covers chunk c of the
// super-block: sub-block 2c in the low nibbles (columns 64c .. 64c+31) and 2c+1 in
// the high nibbles (64c+32 ..). A nibble left at bit position p reads as the float
// 2^23 + q 2^p; one fma with (2^-p, -2^(23-p)) gives q exactly, and a second,
// q * (d sc) - dmin mn, gives the weight with the single rounding of the format's
// formula (d sc q is exact in fp32: an 11-bit fp16 significand times a 6-bit
// scale times a 4-bit quant). So each weight is the oracle's, and the dot product
// has no factored terms that could cancel.
template <int NR, int BT>
QDQ_DEV void dotb_q4k(const uint8_t *const *wrow, int c, const float *xs, float (&out)[NR][BT]) {
    uint4 H[NR], Qa[NR], Qb[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        H[r] = ld4(wrow[r]);
        Qa[r] = ld4(wrow[r] + 16 + 32 * c);
        Qb[r] = ld4(wrow[r] + 32 + 32 * c);
    }
    // q from nibbles at positions (0, 8), (16, 8) [low] and (4, 12) [high]
    const uint64_t P08 = pack2(1.0f, 0.00390625f), N08 = pack2(-kTwo23, -32768.0f);
    const uint64_t P168 = pack2(1.52587890625e-05f, 0.00390625f), N168 = pack2(-128.0f, -32768.0f);
    const uint64_t P412 = pack2(0.0625f, 0.000244140625f), N412 = pack2(-524288.0f, -2048.0f);
    uint64_t DL[NR], ML[NR], DH[NR], MH[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        uint32_t sc2, mn2;
        q4k_pair_fields(H[r].y, H[r].z, H[r].w, c, &sc2, &mn2);
        const float d = half_bits_to_float(H[r].x & 0xFFFF), dmin = half_bits_to_float(H[r].x >> 16);
        const float s_lo = d * (float)(sc2 & 0xFF), s_hi = d * (float)(sc2 >> 8);
        const float m_lo = -(dmin * (float)(mn2 & 0xFF)), m_hi = -(dmin * (float)(mn2 >> 8));
        DL[r] = pack2(s_lo, s_lo);
        ML[r] = pack2(m_lo, m_lo);
        DH[r] = pack2(s_hi, s_hi);
        MH[r] = pack2(m_hi, m_hi);
    }
    uint64_t acc[NR][BT], acc2[NR][BT];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[r][b] = acc2[r][b] = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        uint64_t w0[NR], w1[NR], w2[NR], w3[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t w[8] = {Qa[r].x, Qa[r].y, Qa[r].z, Qa[r].w, Qb[r].x, Qb[r].y, Qb[r].z, Qb[r].w};
            const uint32_t v = w[t], u = v >> 16;
            w0[r] = ffma2(ffma2(bits2(mask_magic<0xFu>(v), mask_magic<0xF00u>(v)), P08, N08), DL[r], ML[r]);
            w1[r] = ffma2(ffma2(bits2(mask_magic<0xF0000u>(v), mask_magic<0xF00u>(u)), P168, N168), DL[r], ML[r]);
            w2[r] = ffma2(ffma2(bits2(mask_magic<0xF0u>(v), mask_magic<0xF000u>(v)), P412, N412), DH[r], MH[r]);
            w3[r] = ffma2(ffma2(bits2(mask_magic<0xF0u>(u), mask_magic<0xF000u>(u)), P412, N412), DH[r], MH[r]);
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            uint64_t xl0, xl1, xh0, xh1;
            xpairs_b(xs, b, 16 * c + t, xl0, xl1);
            xpairs_b(xs, b, 16 * c + 8 + t, xh0, xh1);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                acc[r][b] = ffma2(w1[r], xl1, ffma2(w0[r], xl0, acc[r][b]));
                acc2[r][b] = ffma2(w3[r], xh1, ffma2(w2[r], xh0, acc2[r][b]));
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b)
            out[r][b] = (lo_of(acc[r][b]) + hi_of(acc[r][b])) + (lo_of(acc2[r][b]) + hi_of(acc2[r][b]));
}

// Q6_K, c = 2 h + m (see dot_q6k), NR rows x BT columns.
template <int NR, int BT>
QDQ_DEV void dotb_q6k(const uint8_t *const *wrow, int c, const float *xs, float (&out)[NR][BT]) {
    const int h = c >> 1, m = c & 1;
    uint32_t ql0[NR][4], ql1[NR][4], qh[NR][4], scw[NR][2], dw[NR][1];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const uint8_t *sb = wrow[r];  // 2-byte aligned
        ld_words_a2<4>(sb + 64 * h + 16 * m, ql0[r]);
        ld_words_a2<4>(sb + 64 * h + 32 + 16 * m, ql1[r]);
        ld_words_a2<4>(sb + 128 + 32 * h + 16 * m, qh[r]);
        ld_words_a2<2>(sb + 192 + 8 * h, scw[r]);
        ld_words_a2<1>(sb + 208, dw[r]);
    }
    const uint64_t M32 = bits2(__float_as_uint(kTwo23 + 32.0f), __float_as_uint(kTwo23 + 32.0f));
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) out[r][b] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint64_t acc[NR][BT];
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[r][b] = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            uint64_t p0[NR], p1[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint32_t b6 = q6k_quant_bytes((k & 1) ? ql1[r][t] : ql0[r][t], qh[r][t], k);
                p0[r] = fsub2(bits2(byte_to_magic<0>(b6), byte_to_magic<1>(b6)), M32);
                p1[r] = fsub2(bits2(byte_to_magic<2>(b6), byte_to_magic<3>(b6)), M32);
            }
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                uint64_t x0, x1;
                xpairs_b(xs, b, 32 * h + 8 * k + 4 * m + t, x0, x1);
#pragma unroll
                for (int r = 0; r < NR; ++r) acc[r][b] = ffma2(p1[r], x1, ffma2(p0[r], x0, acc[r][b]));
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int byte = m + 2 * k;
            const uint32_t word = byte < 4 ? scw[r][0] : scw[r][1];
            const float sc = (float)(int)(int8_t)((word >> (8 * (byte & 3))) & 0xFF);
#pragma unroll
            for (int b = 0; b < BT; ++b) out[r][b] += sc * (lo_of(acc[r][b]) + hi_of(acc[r][b]));
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float d = half_bits_to_float(dw[r][0] & 0xFFFF);
#pragma unroll
        for (int b = 0; b < BT; ++b) out[r][b] *= d;
    }
}

// q8_0, NR rows x BT columns; nb = blocks of the slice inside the row.
template <int NR, int BT>
QDQ_DEV void dotb_q8_0(const uint8_t *const *wrow, int c, int nb, const float *xs, float (&out)[NR][BT]) {
    const uint64_t M128 = bits2(__float_as_uint(kTwo23 + 128.0f), __float_as_uint(kTwo23 + 128.0f));
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) out[r][b] = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (2 * c + i >= nb) break;
        uint32_t q[NR][9];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t *base = (const uint32_t *)(wrow[r] + 72 * c + 36 * i);
#pragma unroll
            for (int t = 0; t < 9; ++t) q[r][t] = base[t];
        }
        uint64_t acc[NR][BT];
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[r][b] = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            uint64_t p0[NR], p1[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint32_t v = q[r][1 + t] ^ 0x80808080u;
                p0[r] = fsub2(bits2(byte_to_magic<0>(v), byte_to_magic<1>(v)), M128);
                p1[r] = fsub2(bits2(byte_to_magic<2>(v), byte_to_magic<3>(v)), M128);
            }
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                uint64_t x0, x1;
                xpairs_b(xs, b, 16 * c + 8 * i + t, x0, x1);
#pragma unroll
                for (int r = 0; r < NR; ++r) acc[r][b] = ffma2(p1[r], x1, ffma2(p0[r], x0, acc[r][b]));
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int b = 0; b < BT; ++b)
                out[r][b] += __uint_as_float(q[r][0]) * (lo_of(acc[r][b]) + hi_of(acc[r][b]));
    }
}

// q4_0, NR rows x BT columns (see dot_q4_0 for the nibble layout).
template <int NR, int BT>
QDQ_DEV void dotb_q4_0(const uint8_t *const *wrow, int c, int nb, const float *xs, float (&out)[NR][BT]) {
    const uint64_t C_la = bits2(__float_as_uint(kTwo23 + 8.0f), __float_as_uint(kTwo23 + 2048.0f));
    const uint64_t C_lb = bits2(__float_as_uint(kTwo23 + 524288.0f), __float_as_uint(kTwo23 + 2048.0f));
    const uint64_t C_h = bits2(__float_as_uint(kTwo23 + 128.0f), __float_as_uint(kTwo23 + 32768.0f));
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) out[r][b] = 0.f;
    if (2 * c >= nb) return;  // the slice ends before this lane's blocks
    const bool v1 = 2 * c + 1 < nb;
    uint32_t qs[NR][8];
    float d[NR][2];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        uint32_t w[9];
        if (v1) {
            ld_words_a2<9>(wrow[r] + 36 * c, w);
        } else {
            uint32_t w5[5];
            ld_words_a2<5>(wrow[r] + 36 * c, w5);
#pragma unroll
            for (int i = 0; i < 5; ++i) w[i] = w5[i];
#pragma unroll
            for (int i = 5; i < 9; ++i) w[i] = 0x88888888u;
        }
        d[r][0] = half_bits_to_float(w[0] & 0xFFFF);
        d[r][1] = v1 ? half_bits_to_float(w[4] >> 16) : 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) qs[r][t] = __funnelshift_r(w[t], w[t + 1], 16);
#pragma unroll
        for (int t = 0; t < 4; ++t) qs[r][4 + t] = w[5 + t];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint64_t acc[NR][BT];
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[r][b] = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            uint64_t p0[NR], p1[NR], p2[NR], p3[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint32_t v = qs[r][4 * i + t], u = v >> 16;
                p0[r] = fsub2(bits2(mask_magic<0xFu>(v), mask_magic<0xF00u>(v)), C_la);
                p1[r] = fsub2(bits2(mask_magic<0xF0000u>(v), mask_magic<0xF00u>(u)), C_lb);
                p2[r] = fsub2(bits2(mask_magic<0xF0u>(v), mask_magic<0xF000u>(v)), C_h);
                p3[r] = fsub2(bits2(mask_magic<0xF0u>(u), mask_magic<0xF000u>(u)), C_h);
            }
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                uint64_t xl0, xl1, xh0, xh1;
                xpairs_b(xs, b, 16 * c + 8 * i + t, xl0, xl1);
                xpairs_b(xs, b, 16 * c + 8 * i + 4 + t, xh0, xh1);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    acc[r][b] = ffma2(p3[r], xh1, ffma2(p2[r], xh0, ffma2(p1[r], xl1, ffma2(p0[r], xl0, acc[r][b]))));
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int b = 0; b < BT; ++b) out[r][b] += d[r][i] * (lo_of(acc[r][b]) + hi_of(acc[r][b]));
    }
}

// Shared-memory addresses of a tile's rows: whole rows are contiguous (one
// copy that keeps the source's offset mod 16); padded rows and chunk segments
// sit at a fixed pitch, each keeping its own source offset mod 16.
struct RowGeo {
    uint32_t src_lo;  // low bits of the global address of row 0's first tile byte
    int rb;           // row bytes in global memory
    int pitch;        // stage pitch of padded rows or chunk segments (0: contiguous rows)
};
QDQ_DEV const uint8_t *row_ptr(const uint8_t *stage_p, const RowGeo &g, int r) {
    if (g.pitch == 0) return stage_p + (g.src_lo & 15u) + (uint32_t)(r * g.rb);
    return stage_p + (uint32_t)(r * g.pitch) + ((g.src_lo + (uint32_t)(r * g.rb)) & 15u);
}

// Rows r, r + 8, ... (NR; lane 4 r + c) of one slice against every batch
// column; the row partials go to this warp's column of the level buffer as
// [row][batch column].
template <int TYPE, int NR, int BT>
QDQ_DEV void pass_rows_b(const uint8_t *stage_p, const RowGeo &geo, uint32_t koff, int rp, int left, int r8, int c,
                         int nb, const float *xs, bool fresh, float *mycol) {
    const uint8_t *wrow[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int r = r8 + 8 * i;
        wrow[i] = row_ptr(stage_p, geo, rp + (r < left ? r : left - 1)) + koff;
    }
    float acc[NR][BT];
    if constexpr (TYPE == QDQ_Q4_K) dotb_q4k<NR, BT>(wrow, c, xs, acc);
    else if constexpr (TYPE == QDQ_Q6_K) dotb_q6k<NR, BT>(wrow, c, xs, acc);
    else if constexpr (TYPE == QDQ_Q8_0) dotb_q8_0<NR, BT>(wrow, c, nb, xs, acc);
    else dotb_q4_0<NR, BT>(wrow, c, nb, xs, acc);
#pragma unroll
    for (int i = 0; i < NR; ++i)
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            acc[i][b] += __shfl_xor_sync(0xffffffffu, acc[i][b], 1);
            acc[i][b] += __shfl_xor_sync(0xffffffffu, acc[i][b], 2);
        }
    if (c == 0) {
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int r = r8 + 8 * i;
            if (r < left) {
                float *q = mycol + (rp + r) * BT;
#pragma unroll
                for (int b = 0; b < BT; ++b) q[b] = fresh ? acc[i][b] : q[b] + acc[i][b];
            }
        }
    }
}

template <int TYPE, int BT>
QDQ_DEV void tile_slices_b(const Tile &tl, const DevDesc &d, const uint8_t *stage_p, const RowGeo &geo,
                           const float *xbuf, int cw, int r8, int c, float *mycol) {
    constexpr int QK = (TYPE == QDQ_Q4_K || TYPE == QDQ_Q6_K) ? 256 : 32;
    constexpr int SB = (kSlice / QK) * blk_bytes(TYPE);
    constexpr int KIND = x_kind(TYPE);
    constexpr int NR = Cfg<BT>::kNR;
    const int nk = nkinds(tl.skinds);
    const int slot = __popc(tl.skinds & ((1 << KIND) - 1));
    const int stride = xfloats_per_chunk<BT>(tl.skinds);
    const int nslices = (tl.ccols + kSlice - 1) / kSlice;
    const int k0 = tl.whole ? cw : 8 * tl.chunk + cw;
    const int kend = tl.whole ? nslices : (cw < nslices ? k0 + 1 : k0);
    const int n = tl.nrows;
    bool fresh = tl.first;
    for (int k = k0; k < kend; k += Cfg<BT>::kCW) {
        if (!QDQ_CHECK(&s_status_s1, (k >> 3) >= tl.xw0 && (k >> 3) < tl.xw0 + tl.xwn)) break;  // debug builds
        const float *chunk = xbuf + ((k >> 3) - tl.xw0) * stride;
        const float *xs = chunk + slot * BT * kChunk + (k & 7) * kSlice;
        const int kcols = d.cols - k * kSlice;
        const int nb = (kcols < kSlice ? kcols : kSlice) / QK;
        const uint32_t koff = (uint32_t)(tl.whole ? k : cw) * SB;
        for (int rp = 0; rp < n; rp += 8 * NR) {
            if (NR == 2 && n - rp > 8)
                pass_rows_b<TYPE, NR, BT>(stage_p, geo, koff, rp, n - rp, r8, c, nb, xs, fresh, mycol);
            else
                pass_rows_b<TYPE, 1, BT>(stage_p, geo, koff, rp, n - rp, r8, c, nb, xs, fresh, mycol);
        }
        fresh = false;
    }
    if (fresh && c == 0)  // no slice of this warp in the tile: zero partials
        for (int rr = r8; rr < n; rr += 8)
#pragma unroll
            for (int b = 0; b < BT; ++b) mycol[rr * BT + b] = 0.f;
}

// Batch 1: the tile's work units (row pass, slice) are dealt to the consumer warps
// in turn. A pass covers 8 rows (one per lane group, NR = 1) or 16 (NR = 2, lanes
// also take row r + 8), whichever finishes the tile in fewer unit rounds. A warp
// adds its units' row partials into its own column of the level buffer, which
// the tile's first chunk has zeroed.
template <int TYPE, int NR>
QDQ_DEV void tile_units1_nr(const Tile &tl, const DevDesc &d, const uint8_t *stage_p, const RowGeo &geo,
                            const float *xbuf, int first, int r8, int c, float *mycol, int nslices) {
    constexpr int QK = (TYPE == QDQ_Q4_K || TYPE == QDQ_Q6_K) ? 256 : 32;
    constexpr int SB = (kSlice / QK) * blk_bytes(TYPE);
    constexpr int KIND = x_kind(TYPE);
    constexpr int kCW = Cfg<1>::kCW;
    const int nk = nkinds(tl.skinds);
    const int slot = __popc(tl.skinds & ((1 << KIND) - 1));
    const int stride = xfloats_per_chunk<1>(tl.skinds);
    const int n = tl.nrows, rows_pp = 8 * NR;
    const int npass = (n + rows_pp - 1) / rows_pp;
    // unit u = p * nslices + kk from this warp's first unit, stepped by kCW
    // without divisions in the loop
    int p = first / nslices, kk = first - p * nslices;
    const int dp = kCW / nslices, dk = kCW - dp * nslices;
    for (; p < npass; p += dp, kk += dk) {
        if (kk >= nslices) {
            kk -= nslices;
            ++p;
            if (p >= npass) break;
        }
        const int k = tl.whole ? kk : kSlicesPerChunk * tl.chunk + kk;  // slice of the row
        // debug builds: the slice's x chunk inside the staged window
        if (!QDQ_CHECK(&s_status_s1, (k >> 3) >= tl.xw0 && (k >> 3) < tl.xw0 + tl.xwn)) continue;
        const float *chunk = xbuf + ((k >> 3) - tl.xw0) * stride;
        const float *xs = chunk + slot * kChunk + (k & 7) * kSlice;
        const int kcols = d.cols - k * kSlice;
        const int nb = (kcols < kSlice ? kcols : kSlice) / QK;
        const int rp = p * rows_pp;
        pass_rows_b<TYPE, NR, 1>(stage_p, geo, (uint32_t)kk * SB, rp, n - rp, r8, c, nb, xs, false, mycol);
    }
}

// The units of a level are dealt to the warps round-robin across its tiles: unit
// g of the level (counting this CTA's earlier tiles, `uoff` = their units mod kCW,
// the same in every warp) goes to warp g mod kCW, so the remainders of successive
// tiles fall on different warps and no warp runs more than its share plus one.
template <int TYPE>
QDQ_DEV void tile_units1(const Tile &tl, const DevDesc &d, const uint8_t *stage_p, const RowGeo &geo,
                         const float *xbuf, int cw, int r8, int c, float *mycol, int &uoff) {
    constexpr int kCW = Cfg<1>::kCW;
    const int nslices = (tl.ccols + kSlice - 1) / kSlice;
    // rounds of units each warp runs; a unit of NR rows costs about NR + 1 row
    // units (its fixed part: pointers, scales, the row reduction)
    const int units1 = ((tl.nrows + 7) / 8) * nslices, units2 = ((tl.nrows + 15) / 16) * nslices;
    const int rounds1 = (units1 + kCW - 1) / kCW;
    const int rounds2 = (units2 + kCW - 1) / kCW;
    const int first = (cw - uoff + kCW) % kCW;  // this warp's first unit of the tile
    if (3 * rounds2 <= 2 * rounds1) {
        tile_units1_nr<TYPE, 2>(tl, d, stage_p, geo, xbuf, first, r8, c, mycol, nslices);
        uoff = (uoff + units2) % kCW;
    } else {
        tile_units1_nr<TYPE, 1>(tl, d, stage_p, geo, xbuf, first, r8, c, mycol, nslices);
        uoff = (uoff + units1) % kCW;
    }
}

// ---------------------------------------------------------------------------
// An attention level ("S21 The Capstone: picoLM, in Python", section 4: rope on q
// and k, the fp16 cache written at pos, per-head attention with an online
// softmax and GQA; section 3: interleaved RoPE pairs). Query heads [row0, row0 +
// nrows) of this CTA, by all consumer warps, the x buffer as scratch:
//  * the pair angles pos * f_i formed and reduced by 2 pi in double (four double
//    operations), sincosf of the reduced angle; q_h and k_g turned, k and v
//    rounded to fp16; the group's first head stores them at row pos;
//  * warp w scores the chunks w, w + NCW, ... of eight positions (heads of 32
//    or 64 dimensions: four lanes per position, loads one chunk ahead) or of 32
//    (other heads: lane i takes position c0 + i over the whole head) and adds
//    the chunk's weighted values (lanes over dim pairs), keeping a running
//    maximum, sum and value sum; the current position's key and value come from
//    shared memory;
//  * the warps' states merged in warp order into out[h].
// q, k, v were written by the previous level on other SMs: read through L2.
// ---------------------------------------------------------------------------
constexpr int kAttnMaxD = 256;

// Positions of one head in chunks of eight per warp (chunk c0 = 8 w, 8 (w + NCW),
// ...), for heads of 32 or 64 dimensions. Lane 4 j + e holds the quarter e of
// position c0 + j's key (one or two 16-byte pieces) and value dimensions (2 lane,
// 2 lane + 1) of the chunk's eight positions. The first chunk was copied to this
// warp's shared-memory area by kv_first_copy before the RoPE phase; every later
// chunk is loaded into registers one chunk ahead of its use. Cache rows at or
// after pos are not read: row pos comes from shared memory (kcur, vcur), later
// positions have p = 0 (their copied rows are zero-filled). Online softmax state
// (m, l, a0, a1) as in the per-32 loop.
constexpr int kKVRowBytes = 128;                 // a copied key or value row (64 fp16)
constexpr int kKVAreaBytes = 16 * kKVRowBytes;  // eight key rows, then eight value rows

QDQ_DEV void kv_first_copy(const __half *kc, const __half *vc, int kvd, int g, int D, int pos, int c0, int lane,
                           uint32_t area) {
    // 64 pieces of 16 bytes per matrix: piece p = row p / 8, bytes 16 (p % 8)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int p = lane + 32 * h, row = p >> 3, off = 16 * (p & 7);
        const bool in = c0 + row < pos && off < 2 * D;
        const int64_t e = (int64_t)(in ? c0 + row : 0) * kvd + g * D + off / 2;  // in halves
        const uint32_t n = in ? 16u : 0u;  // zero-fill rows at or after pos
        const uint32_t dk = area + (uint32_t)(row * kKVRowBytes + off);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dk), "l"(kc + e), "r"(n) : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dk + 8 * kKVRowBytes), "l"(vc + e),
                     "r"(n)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int NCW>
QDQ_DEV void attend_chunks8(const __half *kc, const __half *vc, int kvd, int g, int D, int pos, int cw, int lane,
                            const float *qs, const float *kcur, const float *vcur, float inv, const uint8_t *area,
                            float &m, float &l, float &a0, float &a1) {
    const int j = lane >> 2, e4 = lane & 3, dq = D / 4;
    const bool two = dq == 16, vin = 2 * lane < D;
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    const __half2 z2 = __float2half2_rn(0.f);
    uint4 kn0 = z4, kn1 = z4;
    __half2 vn[8];
    auto load = [&](int c0) {
        const int t = c0 + j;
        const bool kin = t < pos;
        const uint4 *kp = reinterpret_cast<const uint4 *>(kc + (int64_t)(kin ? t : 0) * kvd + g * D + e4 * dq);
        kn0 = kin ? __ldcg(kp) : z4;
        kn1 = kin && two ? __ldcg(kp + 1) : z4;
        const __half2 *vp = reinterpret_cast<const __half2 *>(vc + (int64_t)c0 * kvd + g * D) + lane;
#pragma unroll
        for (int u = 0; u < 8; ++u) vn[u] = vin && c0 + u < pos ? __ldcg(vp + (int64_t)u * (kvd / 2)) : z2;
    };
    int c0 = 8 * cw;
    if (c0 <= pos) {  // the first chunk, copied by kv_first_copy
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
        const uint4 *kp = reinterpret_cast<const uint4 *>(area + j * kKVRowBytes + e4 * dq * 2);
        kn0 = kp[0];
        kn1 = two ? kp[1] : z4;
        const __half2 *vp = reinterpret_cast<const __half2 *>(area + 8 * kKVRowBytes) + lane;
#pragma unroll
        for (int u = 0; u < 8; ++u) vn[u] = vin ? vp[u * (kKVRowBytes / 4)] : z2;
    }
    for (; c0 <= pos; c0 += 8 * NCW) {
        const uint4 k0 = kn0, k1 = kn1;
        __half2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = vn[u];
        if (c0 + 8 * NCW <= pos) load(c0 + 8 * NCW);
        const int t = c0 + j, q0 = e4 * dq;
        float dot = 0.f;
        if (t == pos) {
            for (int e = q0; e < q0 + dq; ++e) dot += qs[e] * kcur[e];
        } else {
            const uint32_t w8[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < 4 || two) {
                    const float lo = __half2float(__ushort_as_half((unsigned short)(w8[i] & 0xFFFFu)));
                    const float hi = __half2float(__ushort_as_half((unsigned short)(w8[i] >> 16)));
                    dot += qs[q0 + 2 * i] * lo + qs[q0 + 2 * i + 1] * hi;
                }
            }
        }
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 2);
        const float s = t <= pos ? dot * inv : -INFINITY;
        float cm = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
        const float mn = fmaxf(m, cm);  // finite: position c0 <= pos is in the chunk
        const float scale = expf(m - mn);
        const float p = t <= pos ? expf(s - mn) : 0.f;
        float ps = e4 == 0 ? p : 0.f;  // each position once
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, o);
        l = l * scale + ps;
        a0 *= scale;
        a1 *= scale;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float pu = __shfl_sync(0xFFFFFFFFu, p, 4 * u);
            const float2 f = __half22float2(v[u]);
            a0 += pu * f.x;
            a1 += pu * f.y;
        }
        if (pos < c0 + 8) {  // the current position's value, from shared memory
            const float pu = __shfl_sync(0xFFFFFFFFu, p, 4 * (pos - c0));
            if (vin) {
                a0 += pu * vcur[2 * lane];
                a1 += pu * vcur[2 * lane + 1];
            }
        }
        m = mn;
    }
}

template <int NCW, class A>
QDQ_DEV void attend(const A &a, const DevDesc &d, const DescEx &ex, const Tile &tl, int ctid, int cw, int lane,
                    float *scratch) {
    const int D = d.cols, kvd = d.nkv * D, kv_mul = (int)d.rows / d.nkv, pos = a.attn_pos;
    float *qs = scratch, *kcur = qs + kAttnMaxD, *vcur = kcur + kAttnMaxD;
    float *wm = vcur + kAttnMaxD, *wl = wm + 32, *wacc = wl + 32;  // wacc[NCW][wst]
    const __half *kc = reinterpret_cast<const __half *>(ex.kc), *vc = reinterpret_cast<const __half *>(ex.vc);
    const float inv = 1.0f / sqrtf((float)D);
    const bool vec = (D & 7) == 0, chunks8 = D == 32 || D == 64;
    const int wst = chunks8 ? 64 : kAttnMaxD;
    // chunks of eight: each warp's first chunk is copied here (after wacc)
    uint8_t *kv_area = reinterpret_cast<uint8_t *>(wacc + NCW * 64) + cw * kKVAreaBytes;
    constexpr int kPer2 = kAttnMaxD / 64;
    // debug builds: the heads inside the level's, a position inside the cache
    if (!QDQ_CHECK(&s_status_s1, tl.row0 + tl.nrows <= d.rows && pos >= 0 && D <= kAttnMaxD)) return;
    for (int h = (int)tl.row0; h < (int)tl.row0 + tl.nrows; ++h) {
        const int g = h / kv_mul;
        const bool writer = h % kv_mul == 0;
        // the first chunk's cache rows (written by earlier launches) are in
        // flight during the RoPE phase
        if (chunks8 && 8 * cw <= pos)
            kv_first_copy(kc, vc, kvd, g, D, pos, 8 * cw, lane, (uint32_t)__cvta_generic_to_shared(kv_area));
        for (int i = ctid; i < D / 2; i += NCW * 32) {
            const double th = (double)pos * a.rope_f[i];
            const double turns = rint(th * 0.15915494309189535);
            float sn, cs;
            __sincosf((float)fma(-turns, 6.283185307179586, th), &sn, &cs);  // |angle| <= pi: the fast form is accurate to ~4e-7
            const float qa = __ldcg(d.x + h * D + 2 * i), qb = __ldcg(d.x + h * D + 2 * i + 1);
            qs[2 * i] = qa * cs - qb * sn;
            qs[2 * i + 1] = qa * sn + qb * cs;
            const float ka = __ldcg(ex.x2 + g * D + 2 * i), kb = __ldcg(ex.x2 + g * D + 2 * i + 1);
            const __half k0 = __float2half_rn(ka * cs - kb * sn), k1 = __float2half_rn(ka * sn + kb * cs);
            const __half v0 = __float2half_rn(__ldcg(ex.nw + g * D + 2 * i));
            const __half v1 = __float2half_rn(__ldcg(ex.nw + g * D + 2 * i + 1));
            kcur[2 * i] = __half2float(k0);
            kcur[2 * i + 1] = __half2float(k1);
            vcur[2 * i] = __half2float(v0);
            vcur[2 * i + 1] = __half2float(v1);
            if (writer) {
                const int64_t o = (int64_t)pos * kvd + g * D + 2 * i;
                reinterpret_cast<__half *>(ex.kc)[o] = k0;
                reinterpret_cast<__half *>(ex.kc)[o + 1] = k1;
                reinterpret_cast<__half *>(ex.vc)[o] = v0;
                reinterpret_cast<__half *>(ex.vc)[o + 1] = v1;
            }
        }
        named_bar_sync(kFlushBar, NCW * 32);
        float m = -INFINITY, l = 0.f, acc[2 * kPer2];
#pragma unroll
        for (int j = 0; j < 2 * kPer2; ++j) acc[j] = 0.f;
        if (chunks8)
            attend_chunks8<NCW>(kc, vc, kvd, g, D, pos, cw, lane, qs, kcur, vcur, inv, kv_area,
                                m, l, acc[0], acc[1]);
        for (int c0 = 32 * cw; !chunks8 && c0 <= pos; c0 += 32 * NCW) {
            const int t = c0 + lane;
            float s = -INFINITY;
            if (t <= pos) {
                float dot = 0.f;
                if (t == pos) {
                    for (int e = 0; e < D; ++e) dot += qs[e] * kcur[e];
                } else if (vec) {
                    const uint4 *kr = reinterpret_cast<const uint4 *>(kc + (int64_t)t * kvd + g * D);
                    for (int e = 0; e < D / 8; ++e) {
                        const uint4 u = __ldcg(kr + e);
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float lo = __half2float(__ushort_as_half((unsigned short)(w4[i] & 0xFFFFu)));
                            const float hi = __half2float(__ushort_as_half((unsigned short)(w4[i] >> 16)));
                            dot += qs[8 * e + 2 * i] * lo + qs[8 * e + 2 * i + 1] * hi;
                        }
                    }
                } else {
                    const __half *kr = kc + (int64_t)t * kvd + g * D;
                    for (int e = 0; e < D; ++e) dot += qs[e] * __half2float(kr[e]);
                }
                s = dot * inv;
            }
            float cm = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
            const float mn = fmaxf(m, cm);
            const float scale = expf(m - mn);
            const float p = t <= pos ? expf(s - mn) : 0.f;
            float ps = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, o);
            l = l * scale + ps;
#pragma unroll
            for (int j = 0; j < 2 * kPer2; ++j) acc[j] *= scale;
            const int last = pos - c0 < 31 ? pos - c0 : 31;
            const int nh = c0 + last == pos ? last : last + 1;
            const __half2 *vrow = reinterpret_cast<const __half2 *>(vc + (int64_t)c0 * kvd + g * D);
#pragma unroll 8
            for (int u = 0; u < nh; ++u) {
                const float pu = __shfl_sync(0xFFFFFFFFu, p, u);
#pragma unroll
                for (int j = 0; j < kPer2; ++j) {
                    const int d2 = lane + 32 * j;
                    if (2 * d2 < D) {
                        const float2 f = __half22float2(__ldcg(vrow + (int64_t)u * (kvd / 2) + d2));
                        acc[2 * j] += pu * f.x;
                        acc[2 * j + 1] += pu * f.y;
                    }
                }
            }
            if (nh <= last) {
                const float pu = __shfl_sync(0xFFFFFFFFu, p, last);
#pragma unroll
                for (int j = 0; j < kPer2; ++j) {
                    const int d2 = lane + 32 * j;
                    if (2 * d2 < D) {
                        acc[2 * j] += pu * vcur[2 * d2];
                        acc[2 * j + 1] += pu * vcur[2 * d2 + 1];
                    }
                }
            }
            m = mn;
        }
        if (lane == 0) {
            wm[cw] = m;
            wl[cw] = l;
        }
#pragma unroll
        for (int j = 0; j < kPer2; ++j) {
            const int d2 = lane + 32 * j;
            if (2 * d2 < D) {
                wacc[cw * wst + 2 * d2] = acc[2 * j];
                wacc[cw * wst + 2 * d2 + 1] = acc[2 * j + 1];
            }
        }
        named_bar_sync(kFlushBar, NCW * 32);
        for (int e = ctid; e < D; e += NCW * 32) {  // each warp's factor taken once per output
            float M = -INFINITY, L = 0.f, o = 0.f;
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, wm[w]);
            for (int w = 0; w < NCW; ++w)
                if (wl[w] > 0.f) {
                    const float f = expf(wm[w] - M);
                    L += wl[w] * f;
                    o += wacc[w * wst + e] * f;
                }
            d.y[h * D + e] = o / L;
        }
        // the scratch is reused by the next head, and these stores precede the
        // level's release
        named_bar_sync(kFlushBar, NCW * 32);
    }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
// ATTN: the plan has attention levels (the model's plan). Only that instantiation
// holds the attention code and the rmsnorm folded into the flush: compiled into the
// others, they slowed their GEMV levels by a few per cent.
template <int BT, int MAXD, int MAXL, bool ATTN>
__global__ void __launch_bounds__(Cfg<BT>::kThreads, 1) stream1_kernel(const __grid_constant__ StreamArgs<MAXD, MAXL> a) {
    using SM = Smem<BT, MAXD>;
    constexpr int kBufRows = Cfg<BT>::kBufRows;
    constexpr int kCW = Cfg<BT>::kCW;
    constexpr int kThreads = Cfg<BT>::kThreads;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *xbuf = (float *)(smem + SM::kX);  // x of the staged window, every batch column
    float *part = (float *)(smem + SM::kPart);
    uint64_t *dst = (uint64_t *)(smem + SM::kDst);
    int *dstride = (int *)(smem + SM::kDstStride);
    int64_t *ranges = (int64_t *)(smem + SM::kRanges);
    float *red = (float *)(smem + SM::kRed);
    const uint32_t ring_a = smem_u32(smem);
    const uint32_t full_a = smem_u32(smem + SM::kBars), empty_a = full_a + 8 * kSlots;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, P = gridDim.x;
    int *status = &s_status_s1;
    const bool levels_synced = a.counters != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(full_a + 8 * s, 1);
            mbar_init(empty_a + 8 * s, kCW);
        }
        fence_mbar_init();
    }
    for (int L = 0; L < a.nlevels; ++L)
        for (int g = a.level_start[L] + (int)threadIdx.x; g < a.level_start[L + 1]; g += kThreads)
            cta_rows_by_gemv<ATTN>(a, L, g, cta, P, &ranges[2 * g], &ranges[2 * g + 1]);
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
        int plevel = 0, ptile = 0;  // trace builds: level and tile within it
        walk<BT, ATTN>(
            a, ranges,
            [&](int L) {
                plevel = L;
                ptile = 0;
            },
            [&](const Tile &tl, int, const DevDesc &d) {
                if (tl.attn) return;  // no weights to stream
                if (ptile == 0) S1_TR(plevel, 29);
                const uint32_t bytes = tile_ring_bytes(d, tl.nrows, tl.whole, tl.ccols);
                const uint32_t o = ring_place<BT>(next, bytes);
                // debug builds: the tile lies inside the ring at a 16-byte offset
                const bool placed = QDQ_CHECK(status, o + bytes <= (uint32_t)Cfg<BT>::kRingBytes && (o & 15u) == 0);
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
                const uint32_t nb = placed ? tile_copy(d, tl, stage, bar, kTail) : 0u;
                mbar_arrive_expect_tx(bar, nb);  // releases the tail stores above
                if (placed) tile_copy(d, tl, stage, bar, kBulk);
                if (ptile < 2) S1_TR(plevel, 30 + ptile);
                ++ptile;
                ++t;
            },
            [](int) {});
        (void)plevel;
        for (int i = t - kSlots > 0 ? t - kSlots : 0; i < t; ++i)  // no exit with copies in flight
            mbar_wait(full_a + 8 * (i % kSlots), (i / kSlots) & 1, status);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - kFirstCW;
    const int ctid = (int)threadIdx.x - 32 * kFirstCW;
    const int r8 = lane >> 2, c = lane & 3;
    float *mypart = part + cw * kBufRows * BT;
    int t = 0, cur_e = -1, cur_level = 0, tiles_in_level = 0;
    float row_scale = 1.f;  // 1 / rms of the staged x when its rmsnorm is folded into the flush
    int uoff = 0;           // batch 1: units of the level's earlier tiles, mod the consumer warps
    int buf_rows = 0, rg_base = 0;
    uint32_t ring_next = 0;
    bool had_tiles = false, dep_pending = false, level_staged = false;
    (void)cur_level;

    // Adds the eight warps' partials of every buffered row (warp order) and stores
    // y (adding to it for rows whose earlier columns were stored before).
    // dst[i]: y address of buffer row i; bit 0: add to what y holds (a later
    // column window, or QDQ_Y_ADD), bit 1: the row takes part in the argmax.
    auto flush = [&]() {
        named_bar_sync(kFlushBar, kCW * 32);  // partials and addresses are in place
        unsigned long long best = 0ull;  // argmax candidate: (ordered value, ~row) packed
        for (int i = ctid; BT == 1 && i < buf_rows; i += kCW * 32) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) sum += part[w * kBufRows + i];
            const uint64_t d = dst[i];
            float *yp = (float *)(uintptr_t)(d & ~(uint64_t)3);
            if constexpr (ATTN) {  // 1 / rms of a folded rmsnorm, else 1; its sign: silu
                const float sc = reinterpret_cast<const float *>(dstride)[i];
                sum *= fabsf(sc);
                if (__float_as_uint(sc) >> 31) sum = silu(sum);
            }
            if (d & 1) sum += __ldcg(yp);
            *yp = sum;
            if (d & 2) {
                const unsigned u = __float_as_uint(sum), key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
                const unsigned row = (unsigned)(yp - a.amax_y);
                const unsigned long long k = ((unsigned long long)key << 32) | (0xFFFFFFFFu - row);
                best = k > best ? k : best;
            }
        }
        if (BT == 1 && a.amax_slot != nullptr) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
                best = other > best ? other : best;
            }
            if (lane == 0 && best != 0ull) atomicMax(&a.amax_slot[0], best);
        }
        // batch columns: entry i of a warp's column is (row i / BT, column i % BT)
        for (int i = ctid; BT > 1 && i < buf_rows * BT; i += kCW * 32) {
            const int row = i / BT, b = i - row * BT;
            if (b >= a.batch) continue;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) sum += part[w * kBufRows * BT + i];
            const uint64_t d = dst[row];
            float *yp = (float *)(uintptr_t)(d & ~(uint64_t)3) + (int64_t)b * dstride[row];
            if (d & 1) sum += __ldcg(yp);
            *yp = sum;
        }
        named_bar_sync(kFlushBar, kCW * 32);  // the buffer may be refilled
        buf_rows = 0;
    };

    walk<BT, ATTN>(
        a, ranges,
        [&](int L) {
            cur_level = L;
            tiles_in_level = 0;
            uoff = 0;
            dep_pending = L > 0 && levels_synced;
            level_staged = false;
        },
        [&](const Tile &tl, int e, const DevDesc &d) {
            had_tiles = true;
            if (cw == 0 && lane == 0 && tiles_in_level == 0) S1_TR(cur_level, 4);
            if (dep_pending) {  // wait until every CTA has released the previous level
                if (cw == 0 && lane == 0) {
                    S1_TR(cur_level, 1);
                    wait_counter(&a.counters[cur_level - 1], (unsigned)P, status, kWaitLimitNs);
                    S1_TR(cur_level, 2);
                }
                named_bar_sync(kDepBar, kCW * 32);
                dep_pending = false;
                cur_e = -1;  // x is read again after the dependency
            }
            if constexpr (ATTN) {
                if (tl.attn) {
                    static_assert(3 * kAttnMaxD + 64 + kCW * kAttnMaxD <= Cfg<BT>::kXFloats, "attention scratch");
                    static_assert((3 * kAttnMaxD + 64 + kCW * 64) * 4 + kCW * kKVAreaBytes <= Cfg<BT>::kXFloats * 4 &&
                                      (3 * kAttnMaxD + 64 + kCW * 64) * 4 % 16 == 0,
                                  "attention scratch with the first chunks' copies");
                    attend<kCW>(a, d, a.ex[tl.g], tl, ctid, cw, lane, xbuf);
                    return;
                }
            }
            if (e != cur_e) {
                cur_e = e;
                // the buffer is shared: a later x of the same level waits for every
                // warp to be done with it; then every warp stages its slices
                if (level_staged) named_bar_sync(kFlushBar, kCW * 32);
                float inv[BT];
#pragma unroll
                for (int b = 0; b < BT; ++b) inv[b] = 1.f;
                // rmsnorm at batch 1 with the whole vector in this window: x * w is
                // staged, the lanes add up x^2 on the way, and 1 / rms scales each
                // row's sum at the flush (a scalar factors out of the dot product),
                // so x is read once and no extra barrier is needed
                // (only in the model's instantiation: the extra per-row scale at the
                // flush measured 1 % on the GEMV-only step)
                const bool fold = ATTN && BT == 1 && desc_xop(d) == QDQ_X_RMSNORM && tl.xw0 == 0 &&
                                  tl.xwn * kChunk >= d.cols;
                if (desc_xop(d) == QDQ_X_RMSNORM && !fold)
                    rms_scale<BT>(d, a.ex[tl.g], a.batch, cw, kCW, lane, red, inv);
                float ss = 0.f;
                stage_xb<BT, ATTN>(d, a.ex[tl.g], tl.skinds, a.batch, tl.xw0, tl.xw0 + tl.xwn, cw, kCW, lane, inv, xbuf,
                             fold ? &ss : nullptr);
                if (fold) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
                    if (lane == 0) red[cw] = ss;
                }
                named_bar_sync(kFlushBar, kCW * 32);
                row_scale = 1.f;
                if (fold) {  // every thread adds the warps' sums in warp order
                    float t = 0.f;
                    for (int w = 0; w < kCW; ++w) t += red[w];
                    row_scale = 1.0f / sqrtf(t / (float)d.cols + a.ex[tl.g].eps);
                }
                level_staged = true;
            }
            if (tl.first) {  // a new row group: its rows in the partial buffer
                // Rows whose earlier columns sit in this buffer are stored first.
                if (buf_rows + tl.nrows > kBufRows || (!tl.first_win && buf_rows > 0)) flush();
                rg_base = buf_rows;
                buf_rows += tl.nrows;
                const bool rows_ok = QDQ_CHECK(status, rg_base + tl.nrows <= kBufRows);  // debug builds
                if (cw == 0 && rows_ok)
                    for (int i = lane; i < tl.nrows; i += 32) {
                        dst[rg_base + i] = (uint64_t)(uintptr_t)(d.y + tl.row0 + i) |
                                           ((tl.first_win && desc_yop(d) != QDQ_Y_ADD) ? 0u : 1u) |
                                           (desc_amax(d) ? 2u : 0u);
                        // batch 1: the row's scale at the flush, its sign bit set for a
                        // row stored through silu; wider: y's column stride
                        if constexpr (BT == 1 && ATTN)
                            reinterpret_cast<float *>(dstride)[rg_base + i] =
                                desc_yop(d) == QDQ_Y_SILU ? -row_scale : row_scale;
                        else if constexpr (BT > 1)
                            dstride[rg_base + i] = (int)d.rows;
                    }
                if constexpr (BT == 1) {  // batch 1 adds every unit into the warp's column
                    for (int i = lane; rows_ok && i < tl.nrows; i += 32) mypart[rg_base + i] = 0.f;
                    __syncwarp();
                }
            }
            if (cw == 0 && lane == 0 && tiles_in_level == 0) S1_TR(cur_level, 5);
            if (cw == 0 && lane == 0 && tiles_in_level < 7) S1_TRC(cur_level, 8 + 3 * tiles_in_level);
            const uint32_t toffs = ring_place<BT>(ring_next, tile_ring_bytes(d, tl.nrows, tl.whole, tl.ccols));
            // debug builds: the tile inside the ring, its rows inside the matrix and
            // the row group inside the partial buffer
            const bool tile_ok =
                QDQ_CHECK(status, toffs + tile_ring_bytes(d, tl.nrows, tl.whole, tl.ccols) <= (uint32_t)Cfg<BT>::kRingBytes) &&
                QDQ_CHECK(status, tl.row0 + tl.nrows <= d.rows && rg_base + tl.nrows <= kBufRows);
            const int s = t % kSlots;
            mbar_wait(full_a + 8 * s, (t / kSlots) & 1, status);
            if (cw == 0 && lane == 0 && tiles_in_level == 0) S1_TR(cur_level, 6);
            if (cw == 0 && lane == 0 && tiles_in_level < 7) S1_TRC(cur_level, 9 + 3 * tiles_in_level);
            ++tiles_in_level;

            if (tile_ok) {
                const uint8_t *stage_p = smem + toffs;
                RowGeo geo;
                geo.rb = d.rb;
                if (tl.whole) {
                    geo.src_lo = (uint32_t)(uintptr_t)(d.W + tl.row0 * d.rb);
                    geo.pitch = rows_padded(d) ? whole_pitch(d) : 0;
                } else {
                    geo.src_lo = (uint32_t)(uintptr_t)(d.W + tl.row0 * d.rb + chunk_off(d, tl.chunk));
                    geo.pitch = seg_pitch(seg_bytes(d, tl.ccols));
                }
                float *mycol = mypart + rg_base * BT;
                if constexpr (BT == 1) {
                    switch (d.type) {
                        case QDQ_Q4_K: tile_units1<QDQ_Q4_K>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol, uoff); break;
                        case QDQ_Q6_K: tile_units1<QDQ_Q6_K>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol, uoff); break;
                        case QDQ_Q8_0: tile_units1<QDQ_Q8_0>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol, uoff); break;
                        default: tile_units1<QDQ_Q4_0>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol, uoff); break;
                    }
                } else {
                    switch (d.type) {
                        case QDQ_Q4_K: tile_slices_b<QDQ_Q4_K, BT>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol); break;
                        case QDQ_Q6_K: tile_slices_b<QDQ_Q6_K, BT>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol); break;
                        case QDQ_Q8_0: tile_slices_b<QDQ_Q8_0, BT>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol); break;
                        default: tile_slices_b<QDQ_Q4_0, BT>(tl, d, stage_p, geo, xbuf, cw, r8, c, mycol); break;
                    }
                }
            }
            __syncwarp();
            if (cw == 0 && lane == 0 && tiles_in_level <= 7) S1_TRC(cur_level, 7 + 3 * tiles_in_level);
            if (lane == 0) mbar_arrive(empty_a + 8 * s);
            ++t;
        },
        [&](int L) {
            if (cw == 0 && lane == 0) S1_TR(cur_level, 3);
            if (buf_rows > 0) flush();  // ends with a barrier of the consumer warps after their y stores
            if (cw == 0 && lane == 0) {
                S1_TR(cur_level, 7);
                if (levels_synced) {
                    if (L + 1 < a.nlevels) {
                        // The barrier orders every consumer's y stores before this
                        // release, which makes them visible at GPU scope with the count.
                        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&a.counters[L]) : "memory");
                    } else {
                        __threadfence();
                        const unsigned old = atomicAdd(&a.counters[L], 1u);
                        if (old == (unsigned)P - 1) {  // every CTA has passed every wait: reset for the next run
                            for (int i = 0; i < a.nlevels; ++i) a.counters[i] = 0u;
                            __threadfence();
                        }
                    }
                }
            }
            had_tiles = false;
            dep_pending = false;  // a level without tiles here waits for nothing
        });
    // The argmax: every CTA's candidates are in the slot once it has arrived; the
    // last CTA to arrive writes the winning row and clears the slot for the next
    // run. (The flush that issued this CTA's candidates ended with a barrier of
    // the consumer warps, and the fence orders them before the arrival.)
    if (a.amax_slot != nullptr && cw == 0 && lane == 0) {
        __threadfence();
        if (atomicAdd(&a.amax_slot[1], 1ull) == (unsigned long long)(P - 1)) {
            const unsigned long long v = atomicAdd(&a.amax_slot[0], 0ull);
            *a.amax_out = (long long)(0xFFFFFFFFull - (v & 0xFFFFFFFFull));
            a.amax_slot[0] = 0ull;
            a.amax_slot[1] = 0ull;
            __threadfence();
        }
    }
}

}  // namespace s1

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int BT, int MAXD, int MAXL, bool ATTN = false>
static int launch1(const void *args, int grid, bool cooperative, cudaStream_t stream) {
    auto kern = s1::stream1_kernel<BT, MAXD, MAXL, ATTN>;
    constexpr int smem = s1::Smem<BT, MAXD>::kBytes;
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
            ? cudaLaunchCooperativeKernel((const void *)kern, dim3(grid), dim3(s1::Cfg<BT>::kThreads), params, (size_t)smem,
                                          stream)
            : cudaLaunchKernel((const void *)kern, dim3(grid), dim3(s1::Cfg<BT>::kThreads), params, (size_t)smem, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
}

template <int BT>
static int launch1_bt(const void *args, bool big, bool cooperative, int grid, cudaStream_t stream) {
    return big ? launch1<BT, kMaxPlanDescs, kMaxPlanLevels>(args, grid, cooperative, stream)
               : launch1<BT, kMaxGroupDescs, 1>(args, grid, cooperative, stream);
}

int stream1_launch(const void *args, bool big, bool cooperative, int grid, int bt, bool attn, cudaStream_t stream) {
    if (attn)  // attention levels: batch 1, plan-sized arguments
        return bt == 1 && big ? launch1<1, kMaxPlanDescs, kMaxPlanLevels, true>(args, grid, cooperative, stream)
                              : QDQ_ERR_LIMIT;
    switch (bt) {
        case 1: return launch1_bt<1>(args, big, cooperative, grid, stream);
        case 2: return launch1_bt<2>(args, big, cooperative, grid, stream);
        case 4: return launch1_bt<4>(args, big, cooperative, grid, stream);
        case 8: return launch1_bt<8>(args, big, cooperative, grid, stream);
        default: return QDQ_ERR_LIMIT;
    }
}

int take_status_stream1() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, s_status_s1, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(s_status_s1, &zero, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    return v;
}

}  // namespace qdq
