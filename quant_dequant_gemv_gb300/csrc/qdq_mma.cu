// qdq_mma.cu -- batched dequant-GEMV on the 5th-generation tensor cores (tcgen05).
//
// y[b][r] = sum_c w[r][c] x[b][c] with w = s_g q (+ m_g for Q4_K) inside each scale
// group g of a row (32 weights for Q4_K sub-blocks, q8_0 and q4_0 blocks; 16 for
// Q6_K). Per group the kernel forms Z_g[r][b] = sum_{c in g} q[r][c] x[b][c] on the
// tensor cores and applies the scales on the CUDA cores:
//     y[b][r] = sum_g ( s_g Z_g[r][b] - m_g X_g[b] ),  X_g[b] = sum_{c in g} x[b][c]
// (Q4_K: s = d sc, m = dmin mn; Q6_K: s = d sc, m = 0; q8_0 / q4_0: s = d, m = 0).
// The quants q are small integers, so the A operand (W, M = 128 rows per tile, in
// tensor memory) holds them exactly in bf16; x is split into two bf16 terms,
// x = x_hi + x_lo (round to nearest each), so every product is exact up to the
// rounding of x_lo: |error| <= 2^-17 |w x|, inside the GEMV tolerance for any
// input. Z_g accumulates q x_hi + q x_lo in fp32 tensor memory (two MMAs with
// N = b_pad), one accumulator region per group.
//
// Each CTA splits its own columns of X, sub-chunk by sub-chunk, into the
// MMA's canonical K-major layout in shared memory (and, for Q4_K, the group sums
// X_g), so a call needs no scratch memory and no second launch.
//
// One CTA per SM, 19 warps:
//   warp 0      copies the raw blocks of 128 rows x 256 weights into a ring, with
//               2-D tensor copies of W viewed as [rows / g][g row_bytes]
//               (L2 evict-first);
//   warp 1      owns the tensor memory; its elected lane issues the MMAs;
//   warp 2      reads the fp32 x of each 64-column sub-chunk, splits it into
//               the X slot of the sub-chunk's A stage and (Q4_K) stores the
//               sub-chunk's two group sums in a ring of its own;
//   warps 3-18  turn quants into exact bf16 (a byte permute puts each quant under
//               the bf16 exponent of 128, a bf16 subtraction removes the offset),
//               store them to tensor memory and later read the group
//               accumulators back, adding s_g Z_g (- m_g X_g) into registers.
//               Padded batches up to 32: four groups of four warps (one per
//               tensor-memory lane quarter), group G taking every fourth 64-column
//               sub-chunk whole, so four sub-chunks are in flight. Wider batches:
//               thread (row, run) decodes one 16-quant run of every sub-chunk and
//               reads its accumulator two sub-chunks later.
// Split-K: the CTAs that share a row tile form a thread-block cluster along K.
// Each leaves its partial tile in shared memory and the cluster sums the
// partials through distributed shared memory in rank order, so y is
// overwritten, the result is deterministic, and no global workspace or atomics
// are needed.
//
// Every mbarrier wait is bounded (QDQ_ERR_TIMEOUT in this unit's status word);
// every thread reaches the block and cluster barriers at the end whatever
// happened before, so the kernel always terminates.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {
namespace {

__device__ int s_status_mma;

// Timestamps for performance analysis, compiled in only with -DQDQ_MMA_TRACE:
// slot 0 raw issue (per unit); per decode warp w < 8 and sub-chunk j < 8 at index
// 8 w + j: 2 decode start, 1 stores issued, 3 stores complete; 4 X issue, 5/6 MMA
// saw A/X (per sub-chunk); 7 misc (0 start, 1 accumulator ready, 2 end,
// 3 after the first cluster barrier).
#ifdef QDQ_MMA_TRACE
__device__ unsigned long long *g_mma_trace;
#define MTR(slot, idx)                                                                               \
    do {                                                                                             \
        if (g_mma_trace && (idx) < 64)                                                               \
            g_mma_trace[((size_t)(blockIdx.y * gridDim.x + blockIdx.x) * 8 + (slot)) * 64 + (idx)] = \
                globaltimer_ns();                                                                    \
    } while (0)
#define MTC(slot, idx)                                                                               \
    do {                                                                                             \
        if (g_mma_trace && (idx) < 64)                                                               \
            g_mma_trace[((size_t)(blockIdx.y * gridDim.x + blockIdx.x) * 8 + (slot)) * 64 + (idx)] = \
                (unsigned long long)clock64();                                                       \
    } while (0)
#else
#define MTC(slot, idx) \
    do {               \
    } while (0)
#define MTR(slot, idx) \
    do {               \
    } while (0)
#endif

constexpr int kM = 128;        // rows per tile (MMA M)
constexpr int kUnitK = 256;    // weights per row in one raw stage
constexpr int kSubK = 64;      // weights per row in one A stage (four MMA K-steps of 16)
constexpr int kWarpRaw = 0, kWarpMma = 1, kWarpX = 2, kWarpDec0 = 3, kDecWarps = 16;
constexpr int kThreads = (kWarpDec0 + kDecWarps) * 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxStages = 8;          // per ring (raw, X, D)
constexpr int kAStages = 4;            // A stages in tensor memory (32 columns each)
constexpr int kLag = 2;                // sub-chunks between a decode and its group epilogue
constexpr int kMinSmem = 120 * 1024;   // keeps a second CTA (and its tensor memory) off the SM
constexpr uint32_t kTmemCols = 512;    // A stages in [0, 128), accumulator sets above
constexpr uint32_t kDCol0 = 32 * kAStages;
constexpr uint32_t kSmemBudget = 227u * 1024u;
constexpr uint32_t kFinalOff = 64u * 1024u;  // per-tile result [b][128] after the group combine

// Largest padded batch per launch: the accumulators of kLag + 1 sub-chunks must
// fit in tensor memory (Q6_K has four 16-weight groups per sub-chunk).
__host__ __device__ constexpr int max_bpad(int type) { return type == QDQ_Q6_K ? 32 : 64; }
__host__ __device__ constexpr int groups_per_sub(int type) { return type == QDQ_Q6_K ? 4 : 2; }
// Padded batches up to 32 decode in four groups of four warps, each group taking
// every fourth sub-chunk whole (see the decode warps), when tensor memory holds
// four accumulator sets: four sub-chunks are then in flight, each in its own set.
// The ring then has exactly four sets, so set G belongs to group G alone, and the
// group's parity wait on it cannot confuse two phases.
// Wider batches keep all sixteen warps on every sub-chunk (three sets suffice).
__host__ __device__ constexpr bool rr_groups(int type, int bpad) {
    return bpad <= 32 && groups_per_sub(type) * bpad * 4 <= (int)(512 - 32 * 4);
}
// x_hi and x_lo stacked into one B operand when their accumulator sets still fit.
__host__ __device__ constexpr bool stacked_b(int type, int bpad) {
    return groups_per_sub(type) * 2 * bpad * (rr_groups(type, bpad) ? 4 : 3) <= (int)(512 - 32 * 4);
}

struct MmaArgs {
    const uint8_t *W;   // rows x row_bytes
    const float *x;     // this launch's batch slice of x, [batch][cols] fp32
    float *y;           // [batch][rows]
    int64_t rows, cols, row_bytes;
    int64_t rows_full;  // rows reached through the tensor map (a multiple of g)
    int batch, b_pad, nunits;
    int nraw, nx, nd;   // ring depths: raw W stages, X stages, accumulator sets
    // Raw stage geometry. Rows are grouped in super-rows of g rows, the fewest
    // whose byte length is a multiple of 16, so that W can be described as a 2-D
    // tensor [rows / g][g row_bytes] for the tensor-copy engine. A stage holds
    // nh boxes per region; region m (0 <= m < g) holds rows g s + m, s < 128 / g,
    // each row box_inner bytes, the data starting at the row's 16-byte phase.
    // Rows past rows_full (fewer than g, all in the last tile) are copied row by
    // row into a leftover area at left_off.
    int g, box_inner, kbh, nh;  // kbh: blocks per box
    uint32_t region_bytes, half_bytes, left_off, left_pitch, stage_bytes, pad2;
};

struct Layout {
    uint32_t x, x_stage, sums, xst, bars, tmem_slot, total;
};

// Q4_K group sums of x: a ring of kSumSlots sub-chunks, [slot][group 0..1][b_pad]
// fp32. The X warp fills sub-chunk j only after the MMAs of j - kAStages, which
// came after the epilogue of j - kAStages - (accumulator sets) released its set,
// so a slot is never refilled while its readers may still need it.
constexpr int kSumSlots = 16;

// fp32 x of a sub-chunk as it arrives from global memory: a ring of xstages(b_pad)
// slots, batch row n at n * kXPitch (64 floats and 16 bytes of padding, so that
// eight consecutive rows read 16 bytes each start in eight different bank groups).
// The X warp copies sub-chunk j + xstages - 1 while it splits sub-chunk j, with
// 16-byte asynchronous copies of its own lanes (they take the load path, not the
// copy engine that streams W, so they do not queue behind the weight tiles).
// At 16 padded columns (one item per lane) there is no ring: a lane's loads go
// straight to registers, issued before the wait for the A stage, which measured
// a few per cent faster there; from 32 columns the ring is faster.
constexpr uint32_t kXPitch = 64 * 4 + 16;
__host__ __device__ constexpr int xstages(int b_pad) { return b_pad >= 64 ? 2 : b_pad >= 32 ? 3 : 0; }

__host__ __device__ inline Layout layout_for(uint32_t stage_bytes, int nraw, int nx, int b_pad) {
    Layout L;
    L.x = (uint32_t)nraw * stage_bytes;
    L.x_stage = (uint32_t)(256 * b_pad);  // four K-steps of 2 b_pad rows x 16 bf16
    L.sums = L.x + (uint32_t)nx * L.x_stage;  // nx = kAStages
    L.xst = (L.sums + (uint32_t)(kSumSlots * 2 * b_pad * 4) + 127u) & ~127u;
    L.bars = L.xst + (uint32_t)xstages(b_pad) * (uint32_t)b_pad * kXPitch;
    L.tmem_slot = L.bars + 8u * (6 * kMaxStages + 2 * kAStages + kSumSlots);
    L.total = L.tmem_slot + 16u;
    if (L.total < (uint32_t)kMinSmem) L.total = kMinSmem;
    return L;
}

// ---- tcgen05 / cluster PTX -------------------------------------------------------
QDQ_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
QDQ_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
QDQ_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
QDQ_DEV uint32_t elect_one() {
    uint32_t pred = 0;
    asm volatile("{ .reg .pred P; elect.sync _|P, 0xffffffff; selp.u32 %0, 1, 0, P; }" : "=r"(pred));
    return pred;
}
QDQ_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
QDQ_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) += A (tensor memory) x B (shared memory, by descriptor).
QDQ_DEV void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on the mbarrier once every MMA this thread issued so far has completed.
QDQ_DEV void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

QDQ_DEV void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
QDQ_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

QDQ_DEV void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
QDQ_DEV uint32_t mapa_rank(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
QDQ_DEV float ld_dsmem_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
QDQ_DEV void sts_u8(uint32_t a, uint32_t v) { asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory"); }
QDQ_DEV void sts128(uint32_t a, const uint32_t (&v)[4]) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}
QDQ_DEV uint32_t lds_u16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// Instruction descriptor of kind::f16: fp32 D (bits 4-5 = 1), bf16 A and B (bits
// 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
}
// Shared-memory descriptor of a K-major operand without swizzle: core matrices
// of 8 rows x 16 bytes stored as 128 contiguous bytes; the two core matrices of
// one K-step (K = 16) are 128 bytes apart (leading-dimension offset) and
// successive groups of 8 rows 256 bytes apart (stride-dimension offset).
// Bits 46-47 hold the descriptor version 1; swizzle mode 0 (none).
QDQ_DEV uint64_t make_sdesc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(256u >> 4) << 32) |
           (1ull << 46);
}

// x -> (bf16(x), bf16(x - bf16(x))) for two values; the first value of the pair
// (lower address) goes to the low half of each packed word.
QDQ_DEV void split_pair(uint64_t w2, uint32_t &hi, uint32_t &lo) {
    uint32_t h, l;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi_of(w2)), "f"(lo_of(w2)));
    const uint64_t r = fsub2(w2, bits2(h << 16, h & 0xFFFF0000u));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(hi_of(r)), "f"(lo_of(r)));
    hi = h;
    lo = l;
}

// ---- exact bf16 quants ------------------------------------------------------------
// 0x43 in the high byte of a 16-bit lane is the bf16 exponent of 128 with a unit
// last mantissa place, so a byte v < 128 placed in the low byte reads as the bf16
// 128 + v, exactly; one bf16 subtraction of (128 + offset) then leaves v - offset,
// exactly (a small integer). Selector 0x4140 takes bytes 0 and 1 of w, 0x4342 bytes
// 2 and 3.
QDQ_DEV uint32_t bf16_biased_pair(uint32_t w, uint32_t sel) { return __byte_perm(w, 0x43434343u, sel); }
QDQ_DEV uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
constexpr uint32_t kBf16x2_128 = 0x43004300u;  // (128, 128)
constexpr uint32_t kBf16x2_136 = 0x43084308u;  // (136, 136): q4_0 offset 8
constexpr uint32_t kBf16x2_160 = 0x43204320u;  // (160, 160): Q6_K offset 32

QDQ_DEV uint64_t magic_pair(uint32_t w, int first) {
    return first == 0 ? bits2(byte_to_magic<0>(w), byte_to_magic<1>(w)) : bits2(byte_to_magic<2>(w), byte_to_magic<3>(w));
}

// One run: 16 consecutive quants of one row in a sub-chunk (run r = 2 h + p of four).
// The decoder writes them as eight packed bf16 pairs and returns the run's first
// octet (8 quants) in the sub-chunk and the scale(s) of the run's group.
struct Run {
    uint32_t q[8];
    int octet;
    float s, m;  // w = s q - m
};

// Q4_K: chunk `sub` holds sub-blocks 2 sub (low nibbles) and 2 sub + 1 (high
// nibbles); half h takes bytes 16h..16h+15 of the chunk, p picks the nibble, so
// the group is sub-block 2 sub + p with s = d sc, m = dmin mn. The group is
// recentred (q4k_center): the A operand holds q - rho and the epilogue subtracts
// (m - s rho) X_g, so that both terms stay within a small multiple of sum |w x|.
QDQ_DEV void run_q4k(uint32_t blk, int sub, int h, int p, Run &o) {
    const uint4 H = lds128(blk);
    const uint4 V = lds128(blk + 16 + 32 * sub + 16 * h);
    uint32_t sc2, mn2;
    q4k_pair_fields(H.y, H.z, H.w, sub, &sc2, &mn2);
    o.s = __fmul_rn(half_bits_to_float(H.x & 0xFFFF), (float)((sc2 >> (8 * p)) & 0xFF));
    const float m = __fmul_rn(half_bits_to_float(H.x >> 16), (float)((mn2 >> (8 * p)) & 0xFF));
    const uint32_t rho = (uint32_t)q4k_center(o.s, m, &o.m);
    const uint32_t off16 = 0x4300u + rho;  // the bf16 128 + rho (exact: rho <= 15)
    const uint32_t off = off16 | (off16 << 16);
    const uint32_t v[4] = {V.x, V.y, V.z, V.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t nib = (v[i] >> (4 * p)) & 0x0F0F0F0Fu;
        o.q[2 * i] = bf16x2_sub(bf16_biased_pair(nib, 0x4140), off);
        o.q[2 * i + 1] = bf16x2_sub(bf16_biased_pair(nib, 0x4342), off);
    }
    o.octet = p == 0 ? 2 * h : 4 + 2 * h;
}

// Q6_K: sub-chunk `sub` is half hp = sub / 2 of the block, run k = 2 (sub & 1) + h;
// element 128 hp + 32 k + l (l = 16 p .. 16 p + 15 here) has scale index
// 8 hp + 2 k + p: the run is exactly one scale group. s = d sc, q = q6 - 32.
QDQ_DEV void run_q6k(uint32_t blk, int sub, int h, int p, Run &o) {
    const int hp = sub >> 1, k = 2 * (sub & 1) + h;
    uint32_t ql[4], qh[4];
    lds_words_a2<4>(blk + 64 * hp + 32 * h + 16 * p, ql);  // run k & 1 == h
    lds_words_a2<4>(blk + 128 + 32 * hp + 16 * p, qh);
    const uint32_t scw = lds_u16(blk + 192 + 8 * hp + 2 * k);
    o.s = __fmul_rn(half_bits_to_float(lds_u16(blk + 208)), (float)(int8_t)((scw >> (8 * p)) & 0xFF));
    o.m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t q6 = q6k_quant_bytes(ql[i], qh[i], k);
        o.q[2 * i] = bf16x2_sub(bf16_biased_pair(q6, 0x4140), kBf16x2_160);
        o.q[2 * i + 1] = bf16x2_sub(bf16_biased_pair(q6, 0x4342), kBf16x2_160);
    }
    o.octet = 4 * h + 2 * p;
}

// q8_0 (PETIT): the block at b (block 2 sub + h of the unit, the run's group):
// fp32 d then 32 int8; run p is int8 16p..16p+15. s = d. int8 -> fp32 exactly by
// exponent-field construction, then to bf16 (exact: |q| < 2^8).
QDQ_DEV void run_q8_0(uint32_t b, int h, int p, Run &o) {
    o.s = __uint_as_float(lds32(b));
    o.m = 0.0f;
    const float off = kTwo23 + 128.0f;
    const uint64_t off2 = pack2(off, off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = lds32(b + 4 + 16 * p + 4 * i) ^ 0x80808080u;  // int8 -> q + 128
        const uint64_t f01 = fsub2(magic_pair(v, 0), off2), f23 = fsub2(magic_pair(v, 2), off2);
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.q[2 * i]) : "f"(hi_of(f01)), "f"(lo_of(f01)));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.q[2 * i + 1]) : "f"(hi_of(f23)), "f"(lo_of(f23)));
    }
    o.octet = 4 * h + 2 * p;
}

// q4_0 (PETIT): the block at b (block 2 sub + h of the unit, the run's group):
// fp16 d then 16 bytes whose low nibbles are weights 0-15 and high nibbles weights
// 16-31; run p takes the low (p = 0) or high nibbles. s = d, q = nibble - 8.
QDQ_DEV void run_q4_0(uint32_t b, int h, int p, Run &o) {
    o.s = half_bits_to_float(lds_u16(b));
    o.m = 0.0f;
    uint32_t qs[4];
    lds_words_a2<4>(b + 2, qs);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t nib = (qs[i] >> (4 * p)) & 0x0F0F0F0Fu;
        o.q[2 * i] = bf16x2_sub(bf16_biased_pair(nib, 0x4140), kBf16x2_136);
        o.q[2 * i + 1] = bf16x2_sub(bf16_biased_pair(nib, 0x4342), kBf16x2_136);
    }
    o.octet = 4 * h + 2 * p;
}

template <int TYPE>
QDQ_DEV void decode_run(uint32_t blk, int sub, int h, int p, Run &o) {
    if constexpr (TYPE == QDQ_Q4_K) run_q4k(blk, sub, h, p, o);
    else if constexpr (TYPE == QDQ_Q6_K) run_q6k(blk, sub, h, p, o);
    else if constexpr (TYPE == QDQ_Q8_0) run_q8_0(blk, h, p, o);
    else run_q4_0(blk, h, p, o);
}

// tcgen05.ld of 8 columns of this warp's lanes, with its completion wait.
QDQ_DEV void tmem_ld8(uint32_t ta, uint32_t (&v)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
        : "r"(ta)
        : "memory");
}

// A shared-memory descriptor from its low word (start address, leading offset)
// and high word. Building each MMA's descriptor as a 32-bit add on a
// loop-invariant base keeps the MMA issue at about 10 ns; composing the 64-bit
// value per MMA costs several times that.
QDQ_DEV uint64_t desc_from_words(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}

// A ring slot and its phase, advanced one use at a time (no divisions).
struct Ring {
    int slot = 0, phase = 0, n;
    QDQ_DEV explicit Ring(int n_) : n(n_) {}
    QDQ_DEV void next() {
        if (++slot == n) {
            slot = 0;
            phase ^= 1;
        }
    }
};

QDQ_DEV int unit_k(const MmaArgs &a, int u) {
    const int64_t left = a.cols - (int64_t)u * kUnitK;
    return left < kUnitK ? (int)left : kUnitK;
}

// 2-D tensor copy global -> shared (box at coordinates x, y of the map), counted
// as transaction bytes on the mbarrier, with an L2 cache policy.
QDQ_DEV void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

template <int TYPE, int BP>
__global__ void __launch_bounds__(kThreads, 1)
    mma_gemv_kernel(const MmaArgs a, const __grid_constant__ CUtensorMap wmap) {
    constexpr int kBB = TYPE == QDQ_Q4_K ? 144 : TYPE == QDQ_Q6_K ? 210 : TYPE == QDQ_Q8_0 ? 36 : 18;
    constexpr int kBW = (TYPE == QDQ_Q4_K || TYPE == QDQ_Q6_K) ? 256 : 32;
    constexpr int kUnitBytes = (kUnitK / kBW) * kBB;  // bytes of a full unit of one row
    constexpr int kG = groups_per_sub(TYPE);         // scale groups per sub-chunk
    constexpr int kKbh = TYPE == QDQ_Q8_0 ? 4 : kUnitK / kBW;  // blocks per box row
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int b_pad = BP;  // padded batch (MMA N), a compile-time constant so that every
                               // MMA operand is a fixed offset from a uniform base
    const Layout L = layout_for(a.stage_bytes, a.nraw, a.nx, b_pad);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *status = &s_status_mma;

    const int S = (int)gridDim.x, rank = (int)blockIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * kM;
    const int rows_here = (int)(a.rows - row0 < kM ? a.rows - row0 : kM);
    // rows of this tile reached through the tensor map, and leftover rows
    const int trows = (int)(a.rows_full - row0 <= 0 ? 0 : (a.rows_full - row0 < kM ? a.rows_full - row0 : kM));
    const int nleft = rows_here - trows;
    const int u0 = (int)((int64_t)a.nunits * rank / S), u1 = (int)((int64_t)a.nunits * (rank + 1) / S);
    const int nraw = a.nraw, nd = a.nd;
    // x_hi and x_lo as one stacked B operand (N = 2 b_pad, one MMA per K-step, the
    // two halves summed at read-back) when three sub-chunks of such accumulators fit
    // in tensor memory; otherwise two MMAs per K-step into the same columns
    constexpr bool kStack = stacked_b(TYPE, BP);
    constexpr uint32_t gcols = kStack ? 2 * b_pad : b_pad;  // accumulator columns of one group
    constexpr uint32_t dset = (uint32_t)kG * gcols;         // ... of one sub-chunk
    // sub-chunks of this CTA: four per full unit, fewer for a short last unit; the
    // last sub-chunk of the matrix may have fewer than four K-steps
    const int ns_last = u1 == a.nunits ? (unit_k(a, u1 - 1) + kSubK - 1) / kSubK : kUnitK / kSubK;
    const int J = (u1 - u0 - 1) * (kUnitK / kSubK) + ns_last;
    const int ks_last = u1 == a.nunits ? (unit_k(a, u1 - 1) - kSubK * (ns_last - 1)) / 16 : 4;

    const uint32_t raw_full = sb + L.bars, raw_empty = raw_full + 8 * kMaxStages;
    const uint32_t d_full = raw_empty + 8 * kMaxStages, d_empty = d_full + 8 * kMaxStages;
    const uint32_t a_full = d_empty + 8 * kMaxStages, a_empty = a_full + 8 * kAStages;
    const uint32_t s_full = a_empty + 8 * kAStages;  // Q4_K group sums of a sub-chunk stored
    const uint32_t sums_a = sb + L.sums;
    constexpr int kXs = xstages(BP);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nraw; ++s) {
            mbar_init(raw_full + 8 * s, 1);
            mbar_init(raw_empty + 8 * s, kDecWarps);
        }
        for (int s = 0; s < nd; ++s) {
            mbar_init(d_full + 8 * s, 1);
            mbar_init(d_empty + 8 * s, rr_groups(TYPE, BP) ? 4 : kDecWarps);
        }
        // an A stage is full when its decode warps (16, or the four of a group) have
        // stored its quants and the X warp has stored the sub-chunk's split x
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(a_full + 8 * s, (rr_groups(TYPE, BP) ? 4 : kDecWarps) + 1);
            mbar_init(a_empty + 8 * s, 1);
        }
        for (int s = 0; s < kSumSlots; ++s) mbar_init(s_full + 8 * s, 1);
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(sb + L.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the same value in every lane, and known to the compiler as warp-uniform
    const uint32_t tmem = __shfl_sync(0xFFFFFFFFu, *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot), 0);
    if (threadIdx.x == 0) MTC(7, 0);

    if (warp == kWarpRaw) {
        // ---- raw weight blocks: tensor boxes, plus leftover rows one by one --------
        const uint64_t pol = policy_evict_first();
        const uintptr_t wend16 = (uintptr_t)(a.W + a.rows * a.row_bytes) & ~(uintptr_t)15;
        Ring rs(nraw);
        bool ok = true;
        for (int u = u0, i = 0; u < u1; ++u, ++i, rs.next()) {
            const int s = rs.slot;
            if (i >= nraw) ok = mbar_wait(raw_empty + 8 * s, rs.phase ^ 1, status);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const int uk = unit_k(a, u);
            const int ub = (uk / kBW) * kBB;
            const uint32_t stage = sb + (uint32_t)s * a.stage_bytes;
            const int nh_u = (uk / kBW) > kKbh ? a.nh : 1;  // a short last unit may need one box
            // leftover row lane (< g - 1 of them): 1-D copy from its 16-byte boundary
            uintptr_t src_al = 0;
            uint32_t dst = 0, nbytes = 0;
            if (lane < nleft) {
                const uintptr_t src = (uintptr_t)(a.W + (a.rows_full + lane) * a.row_bytes + (int64_t)u * kUnitBytes);
                const uintptr_t s0 = src & ~(uintptr_t)15, e = src + ub;
                uintptr_t bend = (e + 15) & ~(uintptr_t)15;
                dst = stage + a.left_off + (uint32_t)lane * a.left_pitch;
                if (bend > wend16) {
                    // the matrix's last bytes: bulk up to its last 16-byte boundary,
                    // the rest byte by byte (never read past the end)
                    bend = wend16 > s0 ? wend16 : s0;
                    for (uintptr_t p = bend; p < e; ++p) sts_u8(dst + (uint32_t)(p - s0), *(const uint8_t *)p);
                }
                src_al = s0;
                nbytes = (uint32_t)(bend - s0);
            }
            uint32_t total = nbytes;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
            if (trows > 0) total += (uint32_t)nh_u * a.half_bytes;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(raw_full + 8 * s, total);
                if (trows > 0) {
                    const int y = (int)(row0 / a.g);
                    for (int hb = 0; hb < nh_u; ++hb)
                        for (int m = 0; m < a.g; ++m) {
                            const int64_t off = (int64_t)m * a.row_bytes + (int64_t)u * kUnitBytes + hb * kKbh * kBB;
                            const uint32_t dst_t = stage + hb * a.half_bytes + m * a.region_bytes;
                            // debug builds: a 16-byte aligned destination and x coordinate
                            if (QDQ_CHECK(status, (dst_t & 15u) == 0 && ((off & ~(int64_t)15) & 15) == 0))
                                tma_load_2d(dst_t, &wmap, (int)(off & ~(int64_t)15), y, raw_full + 8 * s, pol);
                        }
                }
            }
            __syncwarp();
            if (nbytes && QDQ_CHECK(status, ((dst | (uint32_t)(uintptr_t)src_al | nbytes) & 15u) == 0))
                bulk_g2s_hint(dst, (const void *)src_al, nbytes, raw_full + 8 * s, pol);
        }
    } else if (warp == kWarpX) {
        // ---- split X. Sub-chunk j's fp32 x (64 columns of each batch row, fewer for
        // a short last sub-chunk) comes from the staging ring (slot j mod kXs, filled
        // kXs - 1 sub-chunks ahead) or, at 16 columns, straight from global memory.
        // The split: item (n, g)
        // of a lane is batch row n and 32-column group g, eight float4 split into
        // bf16 hi + lo and stored in the canonical K-major layout of the X slot (x_hi
        // rows 0..b_pad-1, x_lo rows b_pad..2 b_pad-1; rows past the batch are zero),
        // plus (Q4_K) their sum.
        if constexpr (kXs > 0) {
            Ring rx(kAStages);
            bool ok = true;
            constexpr int kItems = 2 * BP;
            const int nb = a.batch < BP ? a.batch : BP;
            auto sub_ks = [&](int jj) { return jj == J - 1 ? ks_last : 4; };
            // copy sub-chunk jj into its staging slot: 16 bytes per copy, lanes along a
            // row; rows past the batch and columns past a short sub-chunk read as zero
            auto issue = [&](int jj) {
                const int slot = jj % kXs, ks = sub_ks(jj);
                const int64_t c0 = (int64_t)(u0 + jj / (kUnitK / kSubK)) * kUnitK + kSubK * (jj % (kUnitK / kSubK));
                const uint32_t dst0 = sb + L.xst + (uint32_t)(slot * BP) * kXPitch;
    #pragma unroll 4
                for (int i = lane; i < BP * 16; i += 32) {
                    const int n = i >> 4, q = i & 15;
                    const bool in = n < nb && q < 4 * ks;
                    const float *src = a.x + (in ? (int64_t)n * a.cols + c0 + 4 * q : 0);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst0 + (uint32_t)n * kXPitch + 16u * q),
                                 "l"(src), "r"(in ? 16 : 0)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
            // sub-chunk j + kXs - 1 is copied once j has been handed to the MMA, into the
            // slot that j - 1 used
            int jn = 0, j = 0;  // next sub-chunk to copy, to split
            for (; jn < kXs - 1 && jn < J; ++jn) issue(jn);
            for (; j < J && ok; ++j, rx.next()) {
                const int s = rx.slot, ks = sub_ks(j);
                // sub-chunk j's group has landed when at most jn - j - 1 younger ones are pending
                static_assert(xstages(32) <= 3 && xstages(64) <= 3, "wait_group counts below");
                if (jn - j - 1 >= 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
                else asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncwarp();  // every lane's copies of the slot are visible to the warp
                if (j >= kAStages) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_empty + 8 * s, rx.phase ^ 1, status));
                    if (!ok) break;
                }
                const uint32_t xst = sb + L.xst + (uint32_t)((j % kXs) * BP) * kXPitch;
                const uint32_t xslot = sb + L.x + (uint32_t)s * L.x_stage;
                const uint32_t sslot = sums_a + (uint32_t)((j % kSumSlots) * 2 * BP * 4);
    #pragma unroll 1
                for (int it = lane; it < kItems; it += 32) {
                    const int g = it / BP, n = it - g * BP;
                    float4 cur[8];
    #pragma unroll
                    for (int i = 0; i < 8; ++i)
                        cur[i] = lds128f(xst + (uint32_t)n * kXPitch + 128u * g + 16u * i);
    #pragma unroll
                    for (int h = 0; h < 4; ++h) {  // (K-step 2g + (h >> 1), 8-column half h & 1)
                        const int t = 2 * g + (h >> 1), kk = h & 1;
                        if (t < ks) {
                            uint32_t hi[4], lo[4];
                            split_pair(pack2(cur[2 * h].x, cur[2 * h].y), hi[0], lo[0]);
                            split_pair(pack2(cur[2 * h].z, cur[2 * h].w), hi[1], lo[1]);
                            split_pair(pack2(cur[2 * h + 1].x, cur[2 * h + 1].y), hi[2], lo[2]);
                            split_pair(pack2(cur[2 * h + 1].z, cur[2 * h + 1].w), hi[3], lo[3]);
                            const uint32_t blk = xslot + (uint32_t)(t * 64 * BP + kk * 128 + (n & 7) * 16);
                            sts128(blk + (uint32_t)((n >> 3) * 256), hi);
                            sts128(blk + (uint32_t)(((BP + n) >> 3) * 256), lo);
                        }
                    }
                    if constexpr (TYPE == QDQ_Q4_K) {
                        float acc = 0.0f;
    #pragma unroll
                        for (int i = 0; i < 8; ++i) acc += (cur[i].x + cur[i].y) + (cur[i].z + cur[i].w);
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(sslot + (uint32_t)((g * BP + n) * 4)), "f"(acc)
                                     : "memory");
                    }
                }
                // the MMA reads the X slot through the async proxy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    if constexpr (TYPE == QDQ_Q4_K) mbar_arrive(s_full + 8 * (j % kSumSlots));
                    mbar_arrive(a_full + 8 * s);
                }
                if (jn < J) issue(jn++);
            }
            // copies still in flight after a failed wait land before the CTA exits
            asm volatile("cp.async.wait_all;" ::: "memory");
            __syncwarp();
        } else {  // 16 columns: each lane loads its items straight into registers
            Ring rx(kAStages);
            bool ok = true;
            int j = 0;
            constexpr int kItems = 2 * BP;
            auto load_item = [&](int64_t c0, int ks, int it, float4 (&v)[8]) {
                const int g = it / BP, n = it - g * BP;
                const float *src = a.x + (int64_t)n * a.cols + c0 + 32 * g;
    #pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = (n < a.batch && 2 * g + (i >> 2) < ks) ? __ldg(reinterpret_cast<const float4 *>(src) + i)
                                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            };
            for (int u = u0; u < u1 && ok; ++u) {
                const int uk = unit_k(a, u), ns = (uk + kSubK - 1) / kSubK;
                for (int sub = 0; sub < ns && ok; ++sub, ++j, rx.next()) {
                    const int s = rx.slot;
                    const int ks = (uk - kSubK * sub) >= kSubK ? 4 : (uk - kSubK * sub) / 16;
                    const int64_t c0 = (int64_t)u * kUnitK + kSubK * sub;
                    float4 cur[8], nxt[8];
                    load_item(c0, ks, lane, cur);
                    if (j >= kAStages) {
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_empty + 8 * s, rx.phase ^ 1, status));
                        if (!ok) break;
                    }
                    const uint32_t xslot = sb + L.x + (uint32_t)s * L.x_stage;
                    const uint32_t sslot = sums_a + (uint32_t)((j % kSumSlots) * 2 * BP * 4);
    #pragma unroll 1
                    for (int it = lane; it < kItems; it += 32) {
                        if (it + 32 < kItems) load_item(c0, ks, it + 32, nxt);
                        const int g = it / BP, n = it - g * BP;
    #pragma unroll
                        for (int h = 0; h < 4; ++h) {  // (K-step 2g + (h >> 1), 8-column half h & 1)
                            const int t = 2 * g + (h >> 1), kk = h & 1;
                            if (t < ks) {
                                uint32_t hi[4], lo[4];
                                split_pair(pack2(cur[2 * h].x, cur[2 * h].y), hi[0], lo[0]);
                                split_pair(pack2(cur[2 * h].z, cur[2 * h].w), hi[1], lo[1]);
                                split_pair(pack2(cur[2 * h + 1].x, cur[2 * h + 1].y), hi[2], lo[2]);
                                split_pair(pack2(cur[2 * h + 1].z, cur[2 * h + 1].w), hi[3], lo[3]);
                                const uint32_t blk = xslot + (uint32_t)(t * 64 * BP + kk * 128 + (n & 7) * 16);
                                sts128(blk + (uint32_t)((n >> 3) * 256), hi);
                                sts128(blk + (uint32_t)(((BP + n) >> 3) * 256), lo);
                            }
                        }
                        if constexpr (TYPE == QDQ_Q4_K) {
                            float acc = 0.0f;
    #pragma unroll
                            for (int i = 0; i < 8; ++i) acc += (cur[i].x + cur[i].y) + (cur[i].z + cur[i].w);
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sslot + (uint32_t)((g * BP + n) * 4)), "f"(acc)
                                         : "memory");
                        }
    #pragma unroll
                        for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
                    }
                    // the MMA reads the X slot through the async proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (TYPE == QDQ_Q4_K) mbar_arrive(s_full + 8 * (j % kSumSlots));
                        mbar_arrive(a_full + 8 * s);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kWarpMma) {
        // ---- MMA issue: the whole warp runs the loop with warp-uniform operands and
        // one elected lane issues a sub-chunk's MMAs and its two commits in one go,
        // so the descriptors stay in uniform registers (a lone thread issuing from
        // per-thread registers reaches a tenth of the rate).
        // Per K-step t of a sub-chunk: Z_g += q x_hi and Z_g += q x_lo into the
        // accumulator region of t's group.
        const uint32_t idesc = make_idesc(b_pad), idesc2 = make_idesc(2 * b_pad);
        const uint64_t xdesc = make_sdesc(sb + L.x);  // X slot 0, K-step 0
        const uint32_t xdesc_lo = (uint32_t)xdesc, xdesc_hi = (uint32_t)(xdesc >> 32);
        constexpr uint32_t slot_step = (256u * b_pad) >> 4, kstep_step = (64u * b_pad) >> 4;
        constexpr uint32_t lo_step = (32u * b_pad) >> 4;  // the x_lo rows follow the x_hi rows
        int rd_s = 0, rd_p = 0, phase = 0;
        bool ok = true;
        // unrolled over the four A stages: slot s is a compile-time constant
        for (int j0 = 0; j0 < J && ok; j0 += kAStages, phase ^= 1) {
#pragma unroll
            for (int s = 0; s < kAStages; ++s) {
                const int j = j0 + s;
                if (j < J && ok) {
                    if (lane == 0 && j < 8) MTC(7, 16 + j);
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_full + 8 * s, phase, status));
                    if (lane == 0) MTC(5, j);
                    // In four-group mode the set's release needs no wait of its own: group
                    // G releases set j - 4 (the set of j: nd is 4) after its epilogue and
                    // before it decodes sub-chunk j, and the A stage of j is full only
                    // after that decode (its tensor-memory reads are fenced before both
                    // arrivals, in program order).
                    if (!rr_groups(TYPE, BP) && ok && j >= nd)
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(d_empty + 8 * rd_s, rd_p ^ 1, status));
                    if (lane == 0) MTC(6, j);
                    if (ok) {
                        tc_fence_after();
                        if (lane == 0 && j < 8) MTC(7, 40 + j);
                        const int ks = j == J - 1 ? ks_last : 4;
                        const uint32_t dbase = tmem + kDCol0 + (uint32_t)rd_s * dset;
                        if (elect_one()) {
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                if (t < ks) {
                                    const uint32_t bt = xdesc_lo + s * slot_step + t * kstep_step;
                                    const uint32_t dg = dbase + ((kG == 4) ? t : (t >> 1)) * gcols;
                                    const uint32_t acc = (kG == 4) ? 0u : (uint32_t)(t & 1);
                                    if constexpr (kStack) {
                                        mma_ts(dg, tmem + 32u * s + 8 * t, desc_from_words(bt, xdesc_hi), idesc2, acc);
                                    } else {
                                        mma_ts(dg, tmem + 32u * s + 8 * t, desc_from_words(bt, xdesc_hi), idesc, acc);
                                        mma_ts(dg, tmem + 32u * s + 8 * t, desc_from_words(bt + lo_step, xdesc_hi), idesc, 1u);
                                    }
                                }
                            }
                            mma_commit(a_empty + 8 * s);
                            mma_commit(d_full + 8 * rd_s);
                        }
                        __syncwarp();
                        if (lane == 0 && j < 8) MTC(7, 24 + j);
                        if (++rd_s == nd) {
                            rd_s = 0;
                            rd_p ^= 1;
                        }
                    }
                }
            }
        }
    } else if constexpr (rr_groups(TYPE, BP)) {
        // ---- decode in four groups, one warp per tensor-memory lane quarter in each:
        // group G takes sub-chunk G of every unit (j = G, G + 4, ...), decodes all four
        // runs of its rows into A stage G, then waits for that sub-chunk's MMAs and
        // adds s_g Z_g (- m_g X_g) of every scale group into its rows' sums. Four
        // sub-chunks are in flight at once, one per group.
        const int dw = warp - kWarpDec0, G = dw >> 2;
        const int q = warp & 3, rr = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        const int rm = rr < trows ? rr % a.g : 0, rsr = rr < trows ? rr / a.g : 0;
        const uint32_t row_off =
            rr < trows ? (uint32_t)rm * a.region_bytes + (uint32_t)rsr * a.box_inner
                       : (rr < rows_here ? a.left_off + (uint32_t)(rr - trows) * a.left_pitch : 0u);
        const int64_t row_phase = rr < trows ? (int64_t)rm * a.row_bytes : (row0 + rr) * a.row_bytes;
        float yacc[BP];  // this row's sum over the group's sub-chunks, per batch column
#pragma unroll
        for (int i = 0; i < BP; ++i) yacc[i] = 0.0f;
        Ring rs(nraw);
        bool ok = true;
        const bool tr = q == 0 && lane == 0;  // trace builds: one warp per group records
        for (int u = u0; u < u1; ++u, rs.next()) {
            const int sub = G, n = u - u0, j = (kUnitK / kSubK) * n + sub;
            if (tr && n < 8) MTC(0, 8 * G + n);
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(raw_full + 8 * rs.slot, rs.phase, status));
            if (!ok) break;
            const int uk = unit_k(a, u), ns = (uk + kSubK - 1) / kSubK;
            float sg[kG], mg[kG];
            if (sub < ns) {
                const uint32_t stage = sb + (uint32_t)rs.slot * a.stage_bytes + row_off;
                const int64_t unit_phase = row_phase + (int64_t)u * kUnitBytes;
                const uint32_t blk0 = stage + (uint32_t)(unit_phase & 15);
                const uint32_t blk1 = rr < trows ? stage + a.half_bytes + (uint32_t)((unit_phase + kKbh * kBB) & 15)
                                                 : blk0 + kKbh * kBB;
                if (n >= 1) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_empty + 8 * G, (n & 1) ^ 1, status));
                    if (!ok) break;
                    tc_fence_after();
                }
                if (tr && n < 8) MTC(1, 8 * G + n);
#pragma unroll
                for (int run = 0; run < 4; ++run) {
                    const int h = run >> 1, p = run & 1;
                    uint32_t blk = blk0;
                    if constexpr (kBW == 32) {
                        const int kb = 2 * sub + h;
                        blk = (kb < kKbh ? blk0 : blk1) + (uint32_t)(kb & (kKbh - 1)) * kBB;
                    }
                    Run rn;
                    decode_run<TYPE>(blk, sub, h, p, rn);
                    tmem_st8(tl + 32u * G + 4 * rn.octet, rn.q);
                    const int gi = (kG == 4) ? run : (TYPE == QDQ_Q4_K ? p : h);  // the run's scale group
                    sg[gi] = rn.s;
                    mg[gi] = rn.m;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full + 8 * G);
                if (tr && n < 8) MTC(2, 8 * G + n);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty + 8 * rs.slot);  // this group is done with the unit's raw data
            if (sub >= ns) continue;
            // the sub-chunk's accumulators: set j mod nd of the MMA warp's ring, phase
            // j / nd. In this mode nd is 4, so the set's previous phase (sub-chunk
            // j - 4) was this group's own: it saw that phase complete and released
            // the set before decoding j. Its next phase (j + 4) cannot complete before
            // this group releases the set again. So the parity names this phase alone.
            // (Waiting for the previous phase first would be wrong: when this phase
            // has already completed, the barrier sits in the next phase, whose parity
            // is the previous one's, and such a wait could only end with a time-out.)
            const int ds = j % nd, dp = (j / nd) & 1;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(d_full + 8 * ds, dp, status));
            if (!ok) break;
            if (tr && n < 8) MTC(3, 8 * G + n);
            tc_fence_after();
            if constexpr (TYPE == QDQ_Q4_K) {  // the X warp has stored this sub-chunk's group sums
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full + 8 * (j % kSumSlots), (j / kSumSlots) & 1, status));
                if (!ok) break;
            }
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                // a group is present unless a short last sub-chunk (q8_0 / q4_0) ends first
                const bool present = gi * (kSubK / kG) < uk - kSubK * sub;
                const uint32_t dcol = tl + kDCol0 + (uint32_t)ds * dset + gi * gcols;
#pragma unroll
                for (int c8 = 0; c8 < BP / 8; ++c8) {
                    uint32_t v[8];
                    tmem_ld8(dcol + 8 * c8, v);
                    float z[8];
                    if constexpr (kStack) {
                        uint32_t w[8];
                        tmem_ld8(dcol + b_pad + 8 * c8, w);
#pragma unroll
                        for (int t = 0; t < 8; ++t) z[t] = __uint_as_float(v[t]) + __uint_as_float(w[t]);
                    } else {
#pragma unroll
                        for (int t = 0; t < 8; ++t) z[t] = __uint_as_float(v[t]);
                    }
                    if (present) {
                        if constexpr (TYPE == QDQ_Q4_K) {
                            const uint32_t xg = sums_a + (uint32_t)((((j % kSumSlots) * 2 + gi) * b_pad + 8 * c8) * 4);
                            const float4 x0 = lds128f(xg), x1 = lds128f(xg + 16);
                            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int t = 0; t < 8; ++t)
                                yacc[8 * c8 + t] = fmaf(sg[gi], z[t], fmaf(-mg[gi], xv[t], yacc[8 * c8 + t]));
                        } else {
#pragma unroll
                            for (int t = 0; t < 8; ++t) yacc[8 * c8 + t] = fmaf(sg[gi], z[t], yacc[8 * c8 + t]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty + 8 * ds);
            if (tr && n < 8) MTC(4, 8 * G + n);
        }

        // ---- combine the four groups of each row: slot buffer [G][n][128] at offset 0;
        // the first barrier keeps it off raw stages that later groups may still read
        named_bar_sync(1, kDecWarps * 32);
        float *slotbuf = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int b = 0; b < BP; ++b) slotbuf[(G * BP + b) * kM + rr] = yacc[b];
        named_bar_sync(1, kDecWarps * 32);
        if (G == 0) {
            float *fin = reinterpret_cast<float *>(smem + kFinalOff);
            for (int n = 0; n < a.batch; ++n) {
                float v = 0.0f;
#pragma unroll
                for (int g = 0; g < 4; ++g) v += slotbuf[(g * BP + n) * kM + rr];
                if (S == 1) {
                    if (rr < rows_here) a.y[(int64_t)n * a.rows + row0 + rr] = v;
                } else {
                    fin[n * kM + rr] = v;
                }
            }
        }
    } else {
        // ---- decode, and the group epilogue two sub-chunks behind --------------------
        const int dw = warp - kWarpDec0, run = dw >> 2, h = run >> 1, p = run & 1;
        const int q = warp & 3, rr = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        // this row's place in a stage: region m, row s (tensor rows), or the leftover
        // area; rows past the matrix read row 0 of region 0 (their results are dropped)
        const int rm = rr < trows ? rr % a.g : 0, rsr = rr < trows ? rr / a.g : 0;
        const uint32_t row_off =
            rr < trows ? (uint32_t)rm * a.region_bytes + (uint32_t)rsr * a.box_inner
                       : (rr < rows_here ? a.left_off + (uint32_t)(rr - trows) * a.left_pitch : 0u);
        const int64_t row_phase = rr < trows ? (int64_t)rm * a.row_bytes : (row0 + rr) * a.row_bytes;
        // the accumulator this thread reads back: its run's group, and its share of
        // the batch columns (all of them for Q6_K, whose runs are whole groups)
        const int grp = (kG == 4) ? run : (TYPE == QDQ_Q4_K ? p : h);
        const int cw = (kG == 4) ? b_pad : b_pad / 2;
        const int col0 = (kG == 4) ? 0 : (TYPE == QDQ_Q4_K ? h : p) * (b_pad / 2);
        float yacc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) yacc[i] = 0.0f;
        // scales of the last kLag decoded sub-chunks (slot = sub-chunk index & 1)
        // scales of the last two decoded sub-chunks (even / odd sub-chunk index)
        float s_ev = 0.f, m_ev = 0.f, s_od = 0.f, m_od = 0.f;
        int g_ev = -1, g_od = -1;  // global 32-column group of the scale; < 0: group absent
        int rd_s = 0, rd_p = 0, rd_count = 0;
        auto rd_slot = [&]() { return rd_s; };
        auto rd_phase = [&]() { return rd_p; };
        auto rd_next = [&]() {
            if (++rd_s == nd) {
                rd_s = 0;
                rd_p ^= 1;
            }
        };

        // epilogue of one sub-chunk: read back this thread's accumulator columns and
        // add s Z (- m X_g) into yacc; then release the accumulator set
        auto epilogue = [&](float sc, float mn, int gg, int js) -> bool {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(d_full + 8 * rd_slot(), rd_phase(), status))) return false;
            if constexpr (TYPE == QDQ_Q4_K) {  // the X warp has stored sub-chunk js's group sums
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(s_full + 8 * (js % kSumSlots), (js / kSumSlots) & 1, status)))
                    return false;
            }
            if (lane == 0 && dw < 8 && rd_count < 8) MTC(3, dw * 8 + rd_count);
            tc_fence_after();
            const uint32_t dcol = tl + kDCol0 + (uint32_t)rd_slot() * dset + grp * gcols + col0;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                if (8 * c8 < cw) {
                    uint32_t v[8];
                    tmem_ld8(dcol + 8 * c8, v);
                    float z[8];
                    if constexpr (kStack) {
                        uint32_t w[8];
                        tmem_ld8(dcol + b_pad + 8 * c8, w);
#pragma unroll
                        for (int t = 0; t < 8; ++t) z[t] = __uint_as_float(v[t]) + __uint_as_float(w[t]);
                    } else {
#pragma unroll
                        for (int t = 0; t < 8; ++t) z[t] = __uint_as_float(v[t]);
                    }
                    if (gg >= 0) {
                        if constexpr (TYPE == QDQ_Q4_K) {
                            const uint32_t xg =
                                sums_a + (uint32_t)((((js % kSumSlots) * 2 + grp) * b_pad + col0 + 8 * c8) * 4);
                            const float4 x0 = lds128f(xg), x1 = lds128f(xg + 16);
                            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int t = 0; t < 8; ++t) yacc[8 * c8 + t] = fmaf(sc, z[t], fmaf(-mn, xv[t], yacc[8 * c8 + t]));
                        } else {
#pragma unroll
                            for (int t = 0; t < 8; ++t) yacc[8 * c8 + t] = fmaf(sc, z[t], yacc[8 * c8 + t]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty + 8 * rd_slot());
            if (lane == 0 && dw < 8 && rd_count < 8) MTC(4, dw * 8 + rd_count);
            ++rd_count;
            rd_next();
            return true;
        };

        Ring rs(nraw), ra(kAStages);
        bool ok = true;
        int u = u0, sub = 0, ns = 0, uk = 0;
        uint32_t blk0 = 0, blk1 = 0;  // this row's data in the stage: first / second box half
        for (int j = 0; j < J + kLag && ok; ++j) {
            float s_new = 0.f, m_new = 0.f;
            int g_new = -1;
            if (lane == 0 && dw < 8 && j < 8) MTC(0, dw * 8 + j);
            if (j < J) {
                if (sub == 0) {  // a new unit: wait for its raw stage, place this row in it
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(raw_full + 8 * rs.slot, rs.phase, status));
                    if (!ok) break;
                    uk = unit_k(a, u);
                    ns = (uk + kSubK - 1) / kSubK;
                    const uint32_t stage = sb + (uint32_t)rs.slot * a.stage_bytes + row_off;
                    const int64_t unit_phase = row_phase + (int64_t)u * kUnitBytes;
                    if (rr < trows) {
                        blk0 = stage + (uint32_t)(unit_phase & 15);
                        blk1 = stage + a.half_bytes + (uint32_t)((unit_phase + kKbh * kBB) & 15);
                    } else {
                        blk0 = stage + (uint32_t)(unit_phase & 15);
                        blk1 = blk0 + kKbh * kBB;
                    }
                }
                if (j >= kAStages) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_empty + 8 * ra.slot, ra.phase ^ 1, status));
                    if (!ok) break;
                    tc_fence_after();
                }
                if (lane == 0 && dw < 8 && j < 8) MTC(1, dw * 8 + j);
                // the block this thread decodes: the unit's block (K-quants), or
                // block 2 sub + h of the unit (q8_0 / q4_0)
                uint32_t blk = blk0;
                if constexpr (kBW == 32) {
                    const int kb = 2 * sub + h;
                    blk = (kb < kKbh ? blk0 : blk1) + (uint32_t)(kb & (kKbh - 1)) * kBB;
                }
                Run rn;
                decode_run<TYPE>(blk, sub, h, p, rn);
                tmem_st8(tl + 32u * ra.slot + 4 * rn.octet, rn.q);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full + 8 * ra.slot);
                if (lane == 0 && dw < 8 && j < 8) MTC(2, dw * 8 + j);
                ra.next();
                s_new = rn.s;
                m_new = rn.m;
                // the group is present unless a short last sub-chunk (q8_0 / q4_0) ends first
                if (grp * (kSubK / kG) < uk - kSubK * sub) g_new = 8 * u + 2 * sub + grp;
                // advance (u, sub); release the raw stage after its last sub-chunk
                if (++sub == ns) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(raw_empty + 8 * rs.slot);
                    rs.next();
                    sub = 0;
                    ++u;
                }
            }
            const bool odd = j & 1;  // sub-chunk j - 2 has the same parity
            if (j >= kLag) ok = odd ? epilogue(s_od, m_od, g_od, j - kLag) : epilogue(s_ev, m_ev, g_ev, j - kLag);
            if (odd) {
                s_od = s_new;
                m_od = m_new;
                g_od = g_new;
            } else {
                s_ev = s_new;
                m_ev = m_new;
                g_ev = g_new;
            }
        }

        // ---- combine the groups of each row: slot buffer [grp][n][128] at offset 0 --
        float *slotbuf = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
            if (8 * c8 < cw)
#pragma unroll
                for (int t = 0; t < 8; ++t) slotbuf[((grp * b_pad) + col0 + 8 * c8 + t) * kM + rr] = yacc[8 * c8 + t];
        named_bar_sync(1, kDecWarps * 32);
        if (run == 0) {
            float *fin = reinterpret_cast<float *>(smem + kFinalOff);
            for (int n = 0; n < a.batch; ++n) {
                float v = 0.0f;
#pragma unroll
                for (int g = 0; g < kG; ++g) v += slotbuf[(g * b_pad + n) * kM + rr];
                if (S == 1) {
                    if (rr < rows_here) a.y[(int64_t)n * a.rows + row0 + rr] = v;
                } else {
                    fin[n * kM + rr] = v;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (S > 1) {
        // the partials of the cluster's CTAs, summed in rank order
        cluster_sync_all();
        if (threadIdx.x == 0) MTR(7, 3);
        const int r_lo = kM * rank / S, r_hi = kM * (rank + 1) / S, nr = r_hi - r_lo;
        for (int idx = threadIdx.x; idx < a.batch * nr; idx += kThreads) {
            const int n = idx / nr, r = r_lo + idx % nr;
            if (r < rows_here) {
                const uint32_t off = sb + kFinalOff + (uint32_t)(n * kM + r) * 4u;
                float part[kMaxCluster];
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    if (c < S) part[c] = ld_dsmem_f32(mapa_rank(off, (uint32_t)c));
                float acc = 0.0f;
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    if (c < S) acc += part[c];
                a.y[(int64_t)n * a.rows + row0 + r] = acc;
            }
        }
        cluster_sync_all();
    }
    if (threadIdx.x == 0) MTR(7, 2);
}

// ---- host ----------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Raw stage geometry and the tensor map of W viewed as [rows / g][g row_bytes].
int raw_geometry(int type, const void *W, int64_t rows, int64_t cols, MmaArgs &a, CUtensorMap *map) {
    const int bb = qdq_block_bytes(type), bw = qdq_block_weights(type);
    const int64_t ub_full = (int64_t)(kUnitK / bw) * bb;
    a.row_bytes = cols / bw * bb;
    a.g = (int)(16 / gcd64(a.row_bytes, 16));
    a.kbh = type == QDQ_Q8_0 ? 4 : kUnitK / bw;  // a box row holds at most 256 bytes
    a.nh = type == QDQ_Q8_0 ? 2 : 1;
    const int64_t bpb = (int64_t)a.kbh * bb;
    int64_t lead = 0;
    const int64_t nunits = (cols + kUnitK - 1) / kUnitK;
    for (int m = 0; m < a.g; ++m)
        for (int64_t u = 0; u < nunits && u < 16; ++u)
            for (int hb = 0; hb < a.nh; ++hb) lead = std::max(lead, (m * a.row_bytes + u * ub_full + hb * bpb) & 15);
    a.box_inner = (int)((lead + bpb + 15) / 16 * 16);
    if (a.box_inner > 256) return QDQ_ERR_LIMIT;
    a.region_bytes = (uint32_t)((kM / a.g) * a.box_inner);
    a.half_bytes = (uint32_t)(kM * a.box_inner);
    a.left_off = (uint32_t)a.nh * a.half_bytes;
    a.left_pitch = (uint32_t)((ub_full + 15 + 15) / 16 * 16);
    a.rows_full = rows / a.g * a.g;
    const uint32_t left = a.rows_full < rows ? (uint32_t)(a.g - 1) * a.left_pitch : 0u;
    a.stage_bytes = (a.left_off + left + 127u) & ~127u;
    std::memset(map, 0, sizeof(*map));
    if (a.rows_full == 0) return QDQ_OK;  // every row goes the row-by-row way
    if ((int64_t)a.g * a.row_bytes >= ((int64_t)1 << 31)) return QDQ_ERR_LIMIT;
    EncodeTiled enc = encode_fn();
    if (!enc) return QDQ_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)(a.g * a.row_bytes), (cuuint64_t)(a.rows_full / a.g)};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.g * a.row_bytes)};
    const cuuint32_t box[2] = {(cuuint32_t)a.box_inner, (cuuint32_t)(kM / a.g)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QDQ_ERR_CUDA;
    return QDQ_OK;
}

// Ring depths: X stages (at least three, about 64 KiB), accumulator sets in the
// tensor memory above the A stages, and raw stages in the shared memory left.
int ring_depths(int type, MmaArgs &a) {
    const uint32_t x_stage = 256u * (uint32_t)a.b_pad;
    (void)x_stage;
    a.nx = kAStages;  // the X slots travel with the A stages
    const uint32_t dset = (uint32_t)(groups_per_sub(type) * a.b_pad * (stacked_b(type, a.b_pad) ? 2 : 1));
    a.nd = (int)std::min<uint32_t>(kMaxStages, (kTmemCols - kDCol0) / dset);
    if (a.nd < (rr_groups(type, a.b_pad) ? 4 : kLag + 1)) return QDQ_ERR_LIMIT;
    // Four groups keep one sub-chunk each in flight, so more than four sets never
    // fill; with exactly four, each set is only ever used by one group, which then
    // sees every phase of it (the group's accumulator wait relies on this).
    if (rr_groups(type, a.b_pad)) a.nd = 4;
    const Layout L0 = layout_for(a.stage_bytes, 0, a.nx, a.b_pad);
    const uint32_t fixed = L0.tmem_slot + 16u;
    a.nraw = fixed >= kSmemBudget ? 0 : (int)std::min<uint32_t>(kMaxStages, (kSmemBudget - fixed) / a.stage_bytes);
    return a.nraw >= 2 ? QDQ_OK : QDQ_ERR_LIMIT;
}

template <int TYPE, int BP>
int launch_typed(const MmaArgs &a, const CUtensorMap &map, int S, int64_t tiles, cudaStream_t stream) {
    const Layout L = layout_for(a.stage_bytes, a.nraw, a.nx, a.b_pad);
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QDQ_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(mma_gemv_kernel<TYPE, BP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     227 * 1024) != cudaSuccess)
                return QDQ_ERR_CUDA;
            attr_set[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, (unsigned)tiles, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = S > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, mma_gemv_kernel<TYPE, BP>, a, map) != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
}

template <int TYPE>
int max_active_clusters(int S, uint32_t smem) {
    // every b_pad instantiation has the same launch shape; the 16-column one stands for all
    if (cudaFuncSetAttribute(mma_gemv_kernel<TYPE, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mma_gemv_kernel<TYPE, 16>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int TYPE>
int dispatch_bp(const MmaArgs &a, const CUtensorMap &map, int S, int64_t tiles, cudaStream_t stream) {
    switch (a.b_pad) {
        case 16: return launch_typed<TYPE, 16>(a, map, S, tiles, stream);
        case 32: return launch_typed<TYPE, 32>(a, map, S, tiles, stream);
        case 48:
            if constexpr (max_bpad(TYPE) >= 48) return launch_typed<TYPE, 48>(a, map, S, tiles, stream);
            return QDQ_ERR_LIMIT;
        case 64:
            if constexpr (max_bpad(TYPE) >= 64) return launch_typed<TYPE, 64>(a, map, S, tiles, stream);
            return QDQ_ERR_LIMIT;
        default: return QDQ_ERR_LIMIT;
    }
}

int dispatch(int type, const MmaArgs &a, const CUtensorMap &map, int S, int64_t tiles, cudaStream_t stream) {
    switch (type) {
        case QDQ_Q4_K: return dispatch_bp<QDQ_Q4_K>(a, map, S, tiles, stream);
        case QDQ_Q6_K: return dispatch_bp<QDQ_Q6_K>(a, map, S, tiles, stream);
        case QDQ_Q8_0: return dispatch_bp<QDQ_Q8_0>(a, map, S, tiles, stream);
        case QDQ_Q4_0: return dispatch_bp<QDQ_Q4_0>(a, map, S, tiles, stream);
        default: return QDQ_ERR_TYPE;
    }
}

int clusters_fit(int type, int S, uint32_t smem) {
    switch (type) {
        case QDQ_Q4_K: return max_active_clusters<QDQ_Q4_K>(S, smem);
        case QDQ_Q6_K: return max_active_clusters<QDQ_Q6_K>(S, smem);
        case QDQ_Q8_0: return max_active_clusters<QDQ_Q8_0>(S, smem);
        case QDQ_Q4_0: return max_active_clusters<QDQ_Q4_0>(S, smem);
        default: return 0;
    }
}

// Largest cluster size <= want that the device can co-schedule with this much
// shared memory per CTA (cached per device, type and size).
int usable_cluster(int type, int want, uint32_t smem) {
    static std::mutex mu;
    static int cache[64][5][kMaxCluster + 1];  // smallest smem known not to fit, per S (0: none)
    static uint32_t fits[64][5][kMaxCluster + 1];  // largest smem known to fit, per S
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || type < 0 || type > 4) return 1;
    std::lock_guard<std::mutex> lock(mu);
    for (int S = want; S > 1; --S) {
        if (fits[dev][type][S] >= smem) return S;
        if (cache[dev][type][S] != 0 && (uint32_t)cache[dev][type][S] <= smem) continue;
        if (clusters_fit(type, S, smem) >= 1) {
            fits[dev][type][S] = std::max(fits[dev][type][S], smem);
            return S;
        }
        if (cache[dev][type][S] == 0 || (uint32_t)cache[dev][type][S] > smem) cache[dev][type][S] = (int)smem;
    }
    return 1;
}

int mma_cluster_size(int64_t rows, int64_t cols, int sm_count) {
    const int64_t tiles = (rows + kM - 1) / kM;
    const int64_t nunits = (cols + kUnitK - 1) / kUnitK;
    int64_t S = tiles >= sm_count ? 1 : sm_count / tiles;
    S = std::min<int64_t>(S, std::min<int64_t>(kMaxCluster, nunits));
    return (int)std::max<int64_t>(S, 1);
}

}  // namespace

int launch_mma_gemv(int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y, int batch,
                    cudaStream_t stream, int sm_count) {
    if (batch < kMmaMinBatch) return QDQ_ERR_LIMIT;
    RelaxedCaptureScope relaxed;  // first-use setup may run inside a caller's graph capture
    const int64_t tiles = (rows + kM - 1) / kM;
    if (tiles > 65535) return QDQ_ERR_LIMIT;
    if (qdq_block_weights(type) <= 0) return QDQ_ERR_TYPE;
    MmaArgs a;
    std::memset(&a, 0, sizeof(a));
    alignas(64) CUtensorMap map;
    int rc = raw_geometry(type, W, rows, cols, a, &map);
    if (rc) return rc;
    a.W = (const uint8_t *)W;
    a.rows = rows;
    a.cols = cols;
    a.nunits = (int)((cols + kUnitK - 1) / kUnitK);
    const int bmax = max_bpad(type);
    for (int b0 = 0; b0 < batch && rc == QDQ_OK; b0 += bmax) {
        const int bc = batch - b0 < bmax ? batch - b0 : bmax;
        a.batch = bc;
        a.b_pad = (bc + 15) / 16 * 16;
        a.x = x + (int64_t)b0 * cols;
        a.y = y + (int64_t)b0 * rows;
        if ((rc = ring_depths(type, a))) break;
        const uint32_t smem = layout_for(a.stage_bytes, a.nraw, a.nx, a.b_pad).total;
        const int S = usable_cluster(type, mma_cluster_size(rows, cols, sm_count), smem);
        rc = dispatch(type, a, map, S, tiles, stream);
    }
    return rc;
}

#ifdef QDQ_MMA_TRACE
extern "C" void qdq_debug_set_mma_trace(unsigned long long *buf) {
    cudaMemcpyToSymbol(g_mma_trace, &buf, sizeof(buf));
}
#endif

int take_status_mma() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, s_status_mma, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(s_status_mma, &zero, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    return v;
}

}  // namespace qdq
