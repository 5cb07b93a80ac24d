// qdq_stream_common.cuh -- pieces of the streaming (CUDA-core) GEMV kernel that
// the host-side plan packing shares with it: the packed kernel arguments, the
// format constants, the bulk-copy helper and shared-memory read helpers.
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
    // step glue fused into the GEMV (plans only; zero elsewhere): bits 0-3 the x
    // the dot product reads (QDQ_X_*), bits 4-7 how y is written (QDQ_Y_*), bit 8
    // whether the rows take part in the plan's argmax; the operands are in DescEx
    int32_t ops;
    int32_t kinds;  // bit k: the level's x needs swizzled copy kind k (0 plain, 2 q4_0-scaled)
    int32_t nkv;    // attention: KV heads
};
QDQ_DEV int desc_xop(const DevDesc &d) { return d.ops & 15; }
QDQ_DEV int desc_yop(const DevDesc &d) { return (d.ops >> 4) & 15; }
QDQ_DEV bool desc_amax(const DevDesc &d) { return (d.ops >> 8) & 1; }

// Operands of the fused glue and of attention levels, apart from DevDesc so that
// the descriptor the tile walk copies stays small.
struct DescEx {
    const float *x2;  // QDQ_X_SWIGLU: the up input (attention: k)
    const float *nw;  // QDQ_X_RMSNORM: the norm weights (attention: v)
    // attention (type kTypeAttn; x = q, y = the output, rows = query heads, cols =
    // head_dim): the fp16 key / value caches [max_seq][nkv * head_dim]
    uint16_t *kc, *vc;
    float eps;
    int32_t pad;
};

// A plan level that is not a GEMV: the attention block of one position (RoPE,
// fp16 cache append, GQA online softmax), one query head per CTA.
constexpr int kTypeAttn = kPlanAttnType;
constexpr int kMaxRopePairs = 128;

template <int MAXD, int MAXL>
struct StreamArgs {
    int32_t ndesc, nlevels, batch, pad;
    unsigned *counters;
    unsigned long long *trace;  // QDQ_TRACE builds only: per-CTA phase timestamps
    // argmax over the y of the GEMV with amax set (batch 1): packed running
    // maximum and CTA arrivals (plan-owned, zero between runs), the y base its
    // row indices count from, and where the winning index goes
    unsigned long long *amax_slot;
    const float *amax_y;
    long long *amax_out;
    int32_t level_start[MAXL + 1];
    DevDesc d[MAXD];
    DescEx ex[MAXD];
    // attention levels: the position and the pair frequencies base^(-2i/head_dim)
    int32_t attn_pos, pad3;
    double rope_f[kMaxRopePairs];
};

// ---------------------------------------------------------------------------
// Format constants
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int blk_bytes(int t) {
    return t == QDQ_Q4_K ? 144 : t == QDQ_Q6_K ? 210 : t == QDQ_Q8_0 ? 36 : 18;
}
__host__ __device__ constexpr int blk_weights(int t) { return (t == QDQ_Q4_K || t == QDQ_Q6_K) ? 256 : 32; }
// x copy kind a format reads: 0 plain, 2 pre-scaled for q4_0's in-place nibbles.
__host__ __device__ constexpr int x_kind(int t) { return t == QDQ_Q4_0 ? 2 : 0; }

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
// Shared-memory reads of the consumers: plain loads through pointers into the
// dynamic shared array, so the compiler can interleave rows' loads and arithmetic.
// ---------------------------------------------------------------------------
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

// Scale that puts x next to a nibble read at its bit position (see dotb_q4_0): low nibbles of bytes 0..3 of a word sit at bits 0, 8, 16, 8 (the
// last after a 16-bit shift), high nibbles at bits 4, 12, 4, 12.
QDQ_DEV float nibble_scale(bool high, int p) {
    const float lo = p == 0 ? 1.f : p == 2 ? 1.52587890625e-05f : 0.00390625f;
    const float hi = (p & 1) ? 0.000244140625f : 0.0625f;
    return high ? hi : lo;
}

}  // namespace qdq
