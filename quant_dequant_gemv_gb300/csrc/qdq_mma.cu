// qdq_mma.cu -- batched dequant-GEMV on the 5th-generation tensor cores (tcgen05).
//
// y[b][r] = sum_c w[r][c] x[b][c] is computed as D = W X^T: W is the A operand
// (M = 128 rows per tile, K-major, in tensor memory), X the B operand (N = batch,
// K-major, in shared memory), and D is accumulated in fp32 in tensor memory. A
// bf16 operand keeps 8 significant bits, too few for the GEMV tolerance
// 1e-5 * sum|w x|, so both sides are split into two bf16 terms, w = w_hi + w_lo
// and x = x_hi + x_lo with w_hi = bf16(w) and w_lo = bf16(w - w_hi) (round to
// nearest), and w x is taken as w_hi x_hi + w_hi x_lo + w_lo x_hi (the "bf16x3"
// product of Henry, Tang and Heinecke, "Leveraging the bfloat16 Artificial
// Intelligence Datatype For Higher-Precision Computations", ARITH 2019). Each
// term dropped or rounded away is below 2^-16 |w x|. The first two products are
// one MMA with N = 2 b_pad against B = [x_hi; x_lo]; the third is one MMA with
// N = b_pad against x_hi.
//
// X is split once per call by a small kernel into a scratch buffer already in
// the MMA's canonical K-major layout, so every CTA copies its B tiles with one
// bulk copy per 64 columns.
//
// One CTA per SM, 19 warps:
//   warp 0      copies the raw blocks of 128 rows x 256 weights into a ring, with
//               2-D tensor copies of W viewed as [rows / g][g row_bytes]
//               (L2 evict-first);
//   warp 1      owns the tensor memory; its lane 0 issues the MMAs and commits;
//   warp 2      copies the split X of each 64-column sub-chunk into a ring;
//   warps 3-18  decode: thread (row, run) turns a run of 16 consecutive weights
//               of its row per sub-chunk into fp32 with the pages' formulas,
//               splits them and stores the A operand to tensor memory
//               (tcgen05.st). Four warps per row quarter hide each other's
//               latencies.
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
#else
#define MTR(slot, idx) \
    do {               \
    } while (0)
#endif

constexpr int kM = 128;        // rows per tile (MMA M)
constexpr int kUnitK = 256;    // weights per row in one raw stage
constexpr int kSubK = 64;      // weights per row in one A stage (four MMA K-steps of 16)
constexpr int kWarpRaw = 0, kWarpMma = 1, kWarpX = 2, kWarpDec0 = 3, kDecWarps = 16;
constexpr int kThreads = (kWarpDec0 + kDecWarps) * 32;
constexpr int kMaxBPad = 128;
constexpr int kMaxCluster = 8;
constexpr int kMaxStages = 8;          // per ring (raw, X, A)
constexpr int kMinSmem = 120 * 1024;   // keeps a second CTA (and its tensor memory) off the SM
constexpr uint32_t kTmemCols = 512;    // D in columns [0, 2 b_pad), A stages of 64 columns above it
constexpr uint32_t kSmemBudget = 227u * 1024u;

struct MmaArgs {
    const uint8_t *W;   // rows x row_bytes
    const uint8_t *xs;  // split X: per K-step of 16 columns, 2 b_pad rows x 16 bf16 (64 b_pad bytes)
    float *y;           // [batch][rows]
    int64_t rows, cols, row_bytes;
    int64_t rows_full;  // rows reached through the tensor map (a multiple of g)
    int batch, b_pad, nunits;
    int nraw, nx, na;   // ring depths: raw W stages, X stages, A stages (tensor memory)
    // Raw stage geometry. Rows are grouped in super-rows of g rows, the fewest
    // whose byte length is a multiple of 16, so that W can be described as a 2-D
    // tensor [rows / g][g row_bytes] for the tensor-copy engine. A stage holds
    // nh boxes per region; region m (0 <= m < g) holds rows g s + m, s < 128 / g,
    // each row box_inner bytes, the data starting at the row's 16-byte phase.
    // Rows past rows_full (fewer than g, all in the last tile) are copied row by
    // row into a leftover area at left_off.
    int g, box_inner, kbh, nh;  // kbh: blocks per box
    uint32_t region_bytes, half_bytes, left_off, left_pitch, stage_bytes, acol0;
};

struct Layout {
    uint32_t x, x_stage, bars, tmem_slot, total;
};

__host__ __device__ inline Layout layout_for(uint32_t stage_bytes, int nraw, int nx, int b_pad) {
    Layout L;
    L.x = (uint32_t)nraw * stage_bytes;
    L.x_stage = (uint32_t)(256 * b_pad);  // four K-steps of 2 b_pad rows x 16 bf16
    L.bars = (L.x + (uint32_t)nx * L.x_stage + 127u) & ~127u;
    L.tmem_slot = L.bars + 8u * (6 * kMaxStages + 1);
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

// Two 32-lane x 16-column loads and their completion wait in one statement, so
// no use of the registers can be scheduled before the wait.
QDQ_DEV void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
        "[%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
          "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
        : "r"(ta), "r"(tb)
        : "memory");
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
QDQ_DEV uint32_t lds_u16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
QDQ_DEV uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
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

// w -> (bf16(w), bf16(w - bf16(w))) for two weights; the first weight of the pair
// (lower address) goes to the low half of each packed word.
QDQ_DEV void split_pair(uint64_t w2, uint32_t &hi, uint32_t &lo) {
    uint32_t h, l;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi_of(w2)), "f"(lo_of(w2)));
    const uint64_t r = fsub2(w2, bits2(h << 16, h & 0xFFFF0000u));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(hi_of(r)), "f"(lo_of(r)));
    hi = h;
    lo = l;
}

QDQ_DEV uint64_t magic_pair(uint32_t w, int first) {
    return first == 0 ? bits2(byte_to_magic<0>(w), byte_to_magic<1>(w)) : bits2(byte_to_magic<2>(w), byte_to_magic<3>(w));
}

// ---- decoders: one run of 16 consecutive weights of one row ----------------------
// A sub-chunk (64 weights of a row) has four runs; run r = 2 h + p. Each decoder
// fills w2[8] (the run's weights as fp32 pairs) and returns the run's first
// octet (8 weights) within the sub-chunk.

// Q4_K: chunk `sub` holds sub-blocks 2 sub (low nibbles) and 2 sub + 1 (high
// nibbles); half h takes bytes 16h..16h+15 of the chunk, p picks the nibble.
// w = q (d sc) - dmin mn.
QDQ_DEV int decode_q4k(uint32_t blk, int sub, int h, int p, uint64_t (&w2)[8]) {
    const uint4 H = lds128(blk);
    const uint4 V = lds128(blk + 16 + 32 * sub + 16 * h);
    uint32_t sc2, mn2;
    q4k_pair_fields(H.y, H.z, H.w, sub, &sc2, &mn2);
    const float d = half_bits_to_float(H.x & 0xFFFF), dmin = half_bits_to_float(H.x >> 16);
    const float dsc = __fmul_rn(d, (float)((sc2 >> (8 * p)) & 0xFF));
    const float dmn = __fmul_rn(dmin, (float)((mn2 >> (8 * p)) & 0xFF));
    const uint64_t s2 = pack2(dsc, dsc), m2 = pack2(-dmn, -dmn), two23 = pack2(kTwo23, kTwo23);
    const uint32_t v[4] = {V.x, V.y, V.z, V.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t nib = (v[i] >> (4 * p)) & 0x0F0F0F0Fu;
        w2[2 * i] = ffma2(fsub2(magic_pair(nib, 0), two23), s2, m2);
        w2[2 * i + 1] = ffma2(fsub2(magic_pair(nib, 2), two23), s2, m2);
    }
    return p == 0 ? 2 * h : 4 + 2 * h;
}

// Q6_K: sub-chunk `sub` is half hp = sub / 2 of the block, run k = 2 (sub & 1) + h;
// element 128 hp + 32 k + l (l = 16 p .. 16 p + 15 here) has scale index
// 8 hp + 2 k + p. w = (d sc) (q6 - 32).
QDQ_DEV int decode_q6k(uint32_t blk, int sub, int h, int p, uint64_t (&w2)[8]) {
    const int hp = sub >> 1, k = 2 * (sub & 1) + h;
    uint32_t ql[4], qh[4];
    lds_words_a2<4>(blk + 64 * hp + 32 * h + 16 * p, ql);  // run k & 1 == h
    lds_words_a2<4>(blk + 128 + 32 * hp + 16 * p, qh);
    const uint32_t scw = lds_u16(blk + 192 + 8 * hp + 2 * k);
    const float d = half_bits_to_float(lds_u16(blk + 208));
    const float dsc = __fmul_rn(d, (float)(int8_t)((scw >> (8 * p)) & 0xFF));
    const uint64_t s2 = pack2(dsc, dsc);
    const float off = kTwo23 + 32.0f;
    const uint64_t off2 = pack2(off, off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t q6 = q6k_quant_bytes(ql[i], qh[i], k);
        w2[2 * i] = fmul2(fsub2(magic_pair(q6, 0), off2), s2);
        w2[2 * i + 1] = fmul2(fsub2(magic_pair(q6, 2), off2), s2);
    }
    return 4 * h + 2 * p;
}

// q8_0 (PETIT): the block at b (block 2 sub + h of the unit): fp32 d then 32
// int8; run p is int8 16p..16p+15. w = d q.
QDQ_DEV int decode_q8_0(uint32_t b, int h, int p, uint64_t (&w2)[8]) {
    const float d = __uint_as_float(lds32(b));
    const uint64_t d2 = pack2(d, d);
    const float off = kTwo23 + 128.0f;
    const uint64_t off2 = pack2(off, off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = lds32(b + 4 + 16 * p + 4 * i) ^ 0x80808080u;  // int8 -> q + 128
        w2[2 * i] = fmul2(fsub2(magic_pair(v, 0), off2), d2);
        w2[2 * i + 1] = fmul2(fsub2(magic_pair(v, 2), off2), d2);
    }
    return 4 * h + 2 * p;
}

// q4_0 (PETIT): the block at b (block 2 sub + h of the unit): fp16 d then 16
// bytes whose low nibbles are weights 0-15 and high nibbles weights 16-31; run p
// takes the low (p = 0) or high nibbles. w = (q - 8) d.
QDQ_DEV int decode_q4_0(uint32_t b, int h, int p, uint64_t (&w2)[8]) {
    const float d = half_bits_to_float(lds_u16(b));
    uint32_t qs[4];
    lds_words_a2<4>(b + 2, qs);
    const uint64_t d2 = pack2(d, d);
    const float off = kTwo23 + 8.0f;
    const uint64_t off2 = pack2(off, off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t nib = (qs[i] >> (4 * p)) & 0x0F0F0F0Fu;
        w2[2 * i] = fmul2(fsub2(magic_pair(nib, 0), off2), d2);
        w2[2 * i + 1] = fmul2(fsub2(magic_pair(nib, 2), off2), d2);
    }
    return 4 * h + 2 * p;
}

template <int TYPE>
QDQ_DEV int decode_run(uint32_t blk, int sub, int h, int p, uint64_t (&w2)[8]) {
    if constexpr (TYPE == QDQ_Q4_K) return decode_q4k(blk, sub, h, p, w2);
    else if constexpr (TYPE == QDQ_Q6_K) return decode_q6k(blk, sub, h, p, w2);
    else if constexpr (TYPE == QDQ_Q8_0) return decode_q8_0(blk, h, p, w2);
    else return decode_q4_0(blk, h, p, w2);
}

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

template <int TYPE>
__global__ void __launch_bounds__(kThreads, 1)
    mma_gemv_kernel(const MmaArgs a, const __grid_constant__ CUtensorMap wmap) {
    constexpr int kBB = TYPE == QDQ_Q4_K ? 144 : TYPE == QDQ_Q6_K ? 210 : TYPE == QDQ_Q8_0 ? 36 : 18;
    constexpr int kBW = (TYPE == QDQ_Q4_K || TYPE == QDQ_Q6_K) ? 256 : 32;
    constexpr int kUnitBytes = (kUnitK / kBW) * kBB;  // bytes of a full unit of one row
    extern __shared__ __align__(1024) uint8_t smem[];
    const Layout L = layout_for(a.stage_bytes, a.nraw, a.nx, a.b_pad);
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
    const int b_pad = a.b_pad, nraw = a.nraw, nx = a.nx, na = a.na;

    const uint32_t raw_full = sb + L.bars, raw_empty = raw_full + 8 * kMaxStages;
    const uint32_t x_full = raw_empty + 8 * kMaxStages, x_empty = x_full + 8 * kMaxStages;
    const uint32_t a_full = x_empty + 8 * kMaxStages, a_empty = a_full + 8 * kMaxStages;
    const uint32_t acc_full = a_empty + 8 * kMaxStages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nraw; ++s) {
            mbar_init(raw_full + 8 * s, 1);
            mbar_init(raw_empty + 8 * s, kDecWarps);
        }
        for (int s = 0; s < nx; ++s) {
            mbar_init(x_full + 8 * s, 1);
            mbar_init(x_empty + 8 * s, 1);
        }
        for (int s = 0; s < na; ++s) {
            mbar_init(a_full + 8 * s, kDecWarps);
            mbar_init(a_empty + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
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
    if (threadIdx.x == 0) MTR(7, 0);

    if (warp == kWarpRaw) {
        // ---- raw weight blocks: tensor boxes, plus leftover rows one by one --------
        const uint64_t pol = policy_evict_first();
        const uintptr_t wend16 = (uintptr_t)(a.W + a.rows * a.row_bytes) & ~(uintptr_t)15;
        bool ok = true;
        for (int u = u0, i = 0; u < u1; ++u, ++i) {
            const int s = i % nraw;
            if (i >= nraw) ok = mbar_wait(raw_empty + 8 * s, ((i / nraw) + 1) & 1, status);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const int uk = unit_k(a, u);
            const int ub = (uk / kBW) * kBB;
            const uint32_t stage = sb + (uint32_t)s * a.stage_bytes;
            const int nh_u = (uk / kBW) > a.kbh ? a.nh : 1;  // a short last unit may need one box
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
                            const int64_t off = (int64_t)m * a.row_bytes + (int64_t)u * kUnitBytes + hb * a.kbh * kBB;
                            tma_load_2d(stage + hb * a.half_bytes + m * a.region_bytes, &wmap, (int)(off & ~(int64_t)15),
                                        y, raw_full + 8 * s, pol);
                        }
                }
            }
            __syncwarp();
            if (nbytes) bulk_g2s_hint(dst, (const void *)src_al, nbytes, raw_full + 8 * s, pol);
            if (lane == 0) MTR(0, i);
        }
    } else if (warp == kWarpX) {
        // ---- split X, one bulk copy per sub-chunk ----------------------------------
        if (lane == 0) {
            int j = 0;
            bool ok = true;
            for (int u = u0; u < u1 && ok; ++u) {
                const int uk = unit_k(a, u), ns = (uk + kSubK - 1) / kSubK;
                for (int sub = 0; sub < ns; ++sub, ++j) {
                    const int s = j % nx;
                    if (j >= nx && !(ok = mbar_wait(x_empty + 8 * s, ((j / nx) + 1) & 1, status))) break;
                    const int ks = (uk - kSubK * sub) >= kSubK ? 4 : (uk - kSubK * sub) / 16;
                    const int64_t kstep0 = ((int64_t)u * kUnitK + kSubK * sub) / 16;
                    const uint32_t bytes = (uint32_t)(ks * 64 * b_pad);
                    mbar_arrive_expect_tx(x_full + 8 * s, bytes);
                    bulk_g2s(sb + L.x + s * L.x_stage, a.xs + kstep0 * 64 * b_pad, bytes, x_full + 8 * s);
                    MTR(4, j);
                }
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ---- MMA issue: the whole warp runs the loop with warp-uniform operands and
        // one elected lane issues, so the descriptors stay in uniform registers (a
        // lone thread issuing from per-thread registers reaches a tenth of the rate)
        const uint32_t tm = tmem;
        const uint32_t idesc2 = make_idesc(2 * b_pad), idesc1 = make_idesc(b_pad);
        int j = 0;
        bool ok = true;
        for (int u = u0; u < u1 && ok; ++u) {
            const int uk = unit_k(a, u), ns = (uk + kSubK - 1) / kSubK;
            for (int sub = 0; sub < ns; ++sub, ++j) {
                const int sa = j % na, sx = j % nx;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_full + 8 * sa, (j / na) & 1, status));
                if (lane == 0) MTR(5, j);
                ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(x_full + 8 * sx, (j / nx) & 1, status));
                if (lane == 0) MTR(6, j);
                if (!ok) break;
                tc_fence_after();
                const int ks = (uk - kSubK * sub) >= kSubK ? 4 : (uk - kSubK * sub) / 16;
                const uint32_t xbase = sb + L.x + sx * L.x_stage, abase = tm + a.acol0 + 64 * sa;
                for (int t = 0; t < ks; ++t) {
                    const uint64_t bdesc = make_sdesc(xbase + t * 64 * b_pad);
                    const uint32_t acc = (j | t) != 0;
                    if (elect_one()) {
                        mma_ts(tm, abase + 8 * t, bdesc, idesc2, acc);  // hi x [x_hi; x_lo]
                        mma_ts(tm, abase + 32 + 8 * t, bdesc, idesc1, 1u);  // lo x x_hi
                    }
                    __syncwarp();
                }
                if (elect_one()) {
                    mma_commit(a_empty + 8 * sa);
                    mma_commit(x_empty + 8 * sx);
                }
                __syncwarp();
            }
        }
        if (ok && elect_one()) mma_commit(acc_full);
        __syncwarp();
    } else {
        // ---- decode ------------------------------------------------------------------
        const int dw = warp - kWarpDec0, run = dw >> 2, h = run >> 1, p = run & 1;
        const int q = warp & 3, rr = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        // this row's place in a stage: region m, row s (tensor rows), or the leftover
        // area; rows past the matrix read row 0 of region 0 (their results are dropped)
        const int rm = rr < trows ? rr % a.g : 0, rs = rr < trows ? rr / a.g : 0;
        const uint32_t row_off =
            rr < trows ? (uint32_t)rm * a.region_bytes + (uint32_t)rs * a.box_inner
                       : (rr < rows_here ? a.left_off + (uint32_t)(rr - trows) * a.left_pitch : 0u);
        const int64_t row_phase = rr < trows ? (int64_t)rm * a.row_bytes : (row0 + rr) * a.row_bytes;
        bool ok = true;
        int j = 0;
        for (int u = u0, i = 0; u < u1 && ok; ++u, ++i) {
            const int s = i % nraw;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(raw_full + 8 * s, (i / nraw) & 1, status));
            if (!ok) break;
            const uint32_t stage = sb + (uint32_t)s * a.stage_bytes + row_off;
            const int64_t unit_phase = row_phase + (int64_t)u * kUnitBytes;
            const int uk = unit_k(a, u), ns = (uk + kSubK - 1) / kSubK;
            for (int sub = 0; sub < ns; ++sub, ++j) {
                const int sa = j % na;
                if (j >= na) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(a_empty + 8 * sa, ((j / na) + 1) & 1, status));
                    if (!ok) break;
                    tc_fence_after();
                }
                if (lane == 0 && dw < 8 && j < 8) MTR(2, dw * 8 + j);
                // the block this thread decodes: the unit's block (K-quants), or
                // block 2 sub + h of the unit (q8_0 / q4_0)
                const int kb = (kBW == 256) ? 0 : 2 * sub + h;
                uint32_t blk;
                if (rr < trows) {
                    const int hb = kb / a.kbh;
                    const uint32_t lead = (uint32_t)((unit_phase + hb * a.kbh * kBB) & 15);
                    blk = stage + hb * a.half_bytes + lead + (uint32_t)(kb % a.kbh) * kBB;
                } else {
                    blk = stage + (uint32_t)(unit_phase & 15) + (uint32_t)kb * kBB;
                }
                uint64_t w2[8];
                const int o = decode_run<TYPE>(blk, sub, h, p, w2);
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) split_pair(w2[i2], hi[i2], lo[i2]);
                const uint32_t col = tl + a.acol0 + 64 * sa + 4 * o;
                tmem_st8(col, hi);
                tmem_st8(col + 32, lo);
                if (lane == 0 && dw < 8 && j < 8) MTR(1, dw * 8 + j);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && dw < 8 && j < 8) MTR(3, dw * 8 + j);
                if (lane == 0) mbar_arrive(a_full + 8 * sa);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty + 8 * s);
        }

        // ---- epilogue: D (lane = row, column = batch) -> y or the cluster partials --
        if (run == 0) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_full, 0, status));
            if (q == 0 && lane == 0) MTR(7, 1);
            if (ok) {
                tc_fence_after();
                float *red = reinterpret_cast<float *>(smem);
                for (int n0 = 0; n0 < a.batch; n0 += 16) {
                    uint32_t v0[16], v1[16];
                    tmem_ld16x2(tl + n0, tl + b_pad + n0, v0, v1);
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const int n = n0 + t;
                        const float val = __uint_as_float(v0[t]) + __uint_as_float(v1[t]);
                        if (n < a.batch) {
                            if (S == 1) {
                                if (rr < rows_here) a.y[(int64_t)n * a.rows + row0 + rr] = val;
                            } else {
                                red[n * kM + rr] = val;
                            }
                        }
                    }
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
                const uint32_t off = sb + (uint32_t)(n * kM + r) * 4u;
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

// x[batch][cols] fp32 -> the split B operand: for each K-step t of 16 columns a
// block of 2 b_pad rows (x_hi rows 0..b_pad-1, x_lo rows b_pad..2 b_pad-1; rows
// past the batch are zero) in the canonical K-major layout.
__global__ void __launch_bounds__(256) xsplit_kernel(const float *__restrict__ x, int batch, int b_pad, int64_t cols,
                                                     uint8_t *__restrict__ xs) {
    const int64_t total = (cols / 16) * b_pad * 2;  // (K-step, row, octet)
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int kk = (int)(idx & 1);
        const int n = (int)((idx >> 1) % b_pad);
        const int64_t t = (idx >> 1) / b_pad;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (n < batch) {
            const float4 *src = reinterpret_cast<const float4 *>(x + (int64_t)n * cols + 16 * t + 8 * kk);
            v0 = __ldg(src);
            v1 = __ldg(src + 1);
        }
        uint32_t hi[4], lo[4];
        split_pair(pack2(v0.x, v0.y), hi[0], lo[0]);
        split_pair(pack2(v0.z, v0.w), hi[1], lo[1]);
        split_pair(pack2(v1.x, v1.y), hi[2], lo[2]);
        split_pair(pack2(v1.z, v1.w), hi[3], lo[3]);
        uint8_t *blk = xs + t * 64 * b_pad;
        *reinterpret_cast<uint4 *>(blk + (n >> 3) * 256 + kk * 128 + (n & 7) * 16) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(blk + ((b_pad + n) >> 3) * 256 + kk * 128 + (n & 7) * 16) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
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

// Ring depths: X stages (at least three, about 64 KiB), A stages in the tensor
// memory above D, and raw stages in the shared memory that is left.
int ring_depths(MmaArgs &a) {
    const uint32_t x_stage = 256u * (uint32_t)a.b_pad;
    a.nx = (int)std::min<uint32_t>(kMaxStages, std::max<uint32_t>(3u, 65536u / x_stage));
    a.acol0 = (uint32_t)((2 * a.b_pad + 63) / 64 * 64);
    a.na = (int)std::min<uint32_t>(kMaxStages, (kTmemCols - a.acol0) / 64);
    const Layout L0 = layout_for(a.stage_bytes, 0, a.nx, a.b_pad);
    const uint32_t fixed = L0.tmem_slot + 16u;
    a.nraw = fixed >= kSmemBudget ? 0 : (int)std::min<uint32_t>(kMaxStages, (kSmemBudget - fixed) / a.stage_bytes);
    return a.nraw >= 2 ? QDQ_OK : QDQ_ERR_LIMIT;
}

template <int TYPE>
int launch_typed(const MmaArgs &a, const CUtensorMap &map, int S, int64_t tiles, cudaStream_t stream) {
    const Layout L = layout_for(a.stage_bytes, a.nraw, a.nx, a.b_pad);
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QDQ_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(mma_gemv_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    if (cudaLaunchKernelEx(&cfg, mma_gemv_kernel<TYPE>, a, map) != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
}

template <int TYPE>
int max_active_clusters(int S, uint32_t smem) {
    if (cudaFuncSetAttribute(mma_gemv_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
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
    if (cudaOccupancyMaxActiveClusters(&n, mma_gemv_kernel<TYPE>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int dispatch(int type, const MmaArgs &a, const CUtensorMap &map, int S, int64_t tiles, cudaStream_t stream) {
    switch (type) {
        case QDQ_Q4_K: return launch_typed<QDQ_Q4_K>(a, map, S, tiles, stream);
        case QDQ_Q6_K: return launch_typed<QDQ_Q6_K>(a, map, S, tiles, stream);
        case QDQ_Q8_0: return launch_typed<QDQ_Q8_0>(a, map, S, tiles, stream);
        case QDQ_Q4_0: return launch_typed<QDQ_Q4_0>(a, map, S, tiles, stream);
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

// Stream-ordered scratch for the split X, from a pool of this library's own that
// keeps its memory between calls.
int scratch_alloc(void **p, size_t bytes, cudaStream_t stream) {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QDQ_ERR_CUDA;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!pools[dev]) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&pools[dev], &props) != cudaSuccess) {
                cudaGetLastError();
                pools[dev] = nullptr;
                return QDQ_ERR_CUDA;
            }
            uint64_t keep = ~0ull;
            cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
        }
        pool = pools[dev];
    }
    if (cudaMallocFromPoolAsync(p, bytes, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
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
    if (batch <= kStreamMaxBatch) return QDQ_ERR_LIMIT;
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
    const int first = batch < kMaxBPad ? batch : kMaxBPad;
    const int bpad_max = (first + 15) / 16 * 16;
    void *xs = nullptr;
    if ((rc = scratch_alloc(&xs, (size_t)4 * bpad_max * cols, stream))) return rc;
    a.xs = (const uint8_t *)xs;
    for (int b0 = 0; b0 < batch && rc == QDQ_OK; b0 += kMaxBPad) {
        const int bc = batch - b0 < kMaxBPad ? batch - b0 : kMaxBPad;
        a.batch = bc;
        a.b_pad = (bc + 15) / 16 * 16;
        a.y = y + (int64_t)b0 * rows;
        if ((rc = ring_depths(a))) break;
        const uint32_t smem = layout_for(a.stage_bytes, a.nraw, a.nx, a.b_pad).total;
        const int S = usable_cluster(type, mma_cluster_size(rows, cols, sm_count), smem);
        const int64_t work = (cols / 16) * a.b_pad * 2;
        const int grid = (int)std::min<int64_t>((work + 255) / 256, (int64_t)sm_count * 8);
        xsplit_kernel<<<grid, 256, 0, stream>>>(x + (int64_t)b0 * cols, bc, a.b_pad, cols, (uint8_t *)xs);
        if (cudaGetLastError() != cudaSuccess) {
            rc = QDQ_ERR_CUDA;
            break;
        }
        rc = dispatch(type, a, map, S, tiles, stream);
    }
    if (cudaFreeAsync(xs, stream) != cudaSuccess) {
        cudaGetLastError();
        if (rc == QDQ_OK) rc = QDQ_ERR_CUDA;
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
