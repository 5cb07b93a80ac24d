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

#include "qdq_stream_common.cuh"

namespace qdq {

static __device__ int s_status_stream;

// Phase timestamps for performance analysis, compiled in only with -DQDQ_TRACE:
// trace[(cta * nlevels + level) * 32 + slot] = %globaltimer (QDQ_TR) or the SM's
// clock64 (QDQ_TRC, for the per-tile phases of the first consumer warp).
#ifdef QDQ_TRACE
#define QDQ_TR(L, slot)                                                                                 \
    do {                                                                                                \
        if (a.trace) a.trace[((size_t)blockIdx.x * a.nlevels + (L)) * 32 + (slot)] = globaltimer_ns(); \
    } while (0)
#define QDQ_TRC(L, slot)                                                                                    \
    do {                                                                                                    \
        if (a.trace) a.trace[((size_t)blockIdx.x * a.nlevels + (L)) * 32 + (slot)] = (uint64_t)clock64(); \
    } while (0)
#else
#define QDQ_TR(L, slot) \
    do {                \
    } while (0)
#define QDQ_TRC(L, slot) \
    do {                 \
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

template <int BT, int MAXD>
constexpr int smem_bytes() {
    return Cfg<BT>::kStages * kStageBytes + 2 * Cfg<BT>::kXBytes + 2 * Cfg<BT>::kXSumBytes + MAXD * 16 +
           (2 * Cfg<BT>::kStages + 6) * 8;
}

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
            if (cw == 0 && lane == 0 && tiles_in_level < 7) QDQ_TRC(cur_level, 8 + 3 * tiles_in_level);
            const int s = t % NST;
            mbar_wait(full_a + 8 * s, (t / NST) & 1, status);
            if (cw == 0 && lane == 0 && tiles_in_level == 0) QDQ_TR(cur_level, 6);
            if (cw == 0 && lane == 0 && tiles_in_level < 7) QDQ_TRC(cur_level, 9 + 3 * tiles_in_level);
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
            if (cw == 0 && lane == 0 && tiles_in_level <= 7) QDQ_TRC(cur_level, 7 + 3 * tiles_in_level);
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
    if (p->bt == 1) return stream1_launch(p->args, p->big, p->cooperative, p->grid, stream);
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
