// qdq_dequant.cu -- standalone dequantisation: blocks -> fp32, bit-exact.
//
// "S21 The Capstone: picoLM, in Python", section 2 (dequantize_q4_K: raw blocks
// and a count n in, n floats out); "PicoLM Q6_K quantisation bug"
// (dequantize_row_q6_K with the is + l/16 scale index); "PETIT" (q8_0, q4_0).
//
// One thread produces 4 consecutive weights and writes them with one 16-byte
// store, so a warp writes 512 contiguous bytes per instruction. The kernel is
// bound by the fp32 write (4 bytes out per 0.56-1.13 bytes in).
#include <cstdint>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return (uint32_t)__ldg((const unsigned short *)p);
}
__device__ __forceinline__ uint32_t ldg_u32(const uint8_t *p) { return __ldg((const unsigned int *)p); }
// 4 bytes at a 2-byte-aligned address
__device__ __forceinline__ uint32_t ldg_u32_a2(const uint8_t *p) { return ldg_u16(p) | (ldg_u16(p + 2) << 16); }

template <int TYPE>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ blocks, int64_t nquads,
                                                      float *__restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < nquads; t += stride) {
        float4 v;
        if constexpr (TYPE == QDQ_Q4_K) {
            const int64_t b = t >> 6;          // 64 quads per 256-weight block
            const int e0 = (int)(t & 63) * 4;  // first weight of the quad
            const uint8_t *blk = blocks + b * 144;
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
        } else if constexpr (TYPE == QDQ_Q6_K) {
            const int64_t b = t >> 6;
            const int e0 = (int)(t & 63) * 4;
            const uint8_t *blk = blocks + b * 210;  // 2-byte aligned
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
        } else if constexpr (TYPE == QDQ_Q8_0) {
            const int64_t b = t >> 3;  // 8 quads per 32-weight block
            const int e0 = (int)(t & 7) * 4;
            const uint8_t *blk = blocks + b * 36;  // 4-byte aligned
            const float d = __uint_as_float(ldg_u32(blk));
            const uint32_t q = ldg_u32(blk + 4 + e0);
            v.x = q8_0_weight(d, (int)(int8_t)(q & 0xFF));
            v.y = q8_0_weight(d, (int)(int8_t)((q >> 8) & 0xFF));
            v.z = q8_0_weight(d, (int)(int8_t)((q >> 16) & 0xFF));
            v.w = q8_0_weight(d, (int)(int8_t)(q >> 24));
        } else {  // QDQ_Q4_0
            const int64_t b = t >> 3;
            const int e0 = (int)(t & 7) * 4;
            const uint8_t *blk = blocks + b * 18;  // 2-byte aligned
            const float d = half_bits_to_float(ldg_u16(blk));
            uint32_t q = ldg_u32_a2(blk + 2 + (e0 & 15));
            if (e0 >= 16) q >>= 4;
            v.x = q4_0_weight(d, (int)(q & 15));
            v.y = q4_0_weight(d, (int)((q >> 8) & 15));
            v.z = q4_0_weight(d, (int)((q >> 16) & 15));
            v.w = q4_0_weight(d, (int)((q >> 24) & 15));
        }
        reinterpret_cast<float4 *>(out)[t] = v;
    }
}

int launch_dequant(int type, const void *blocks, int64_t n, float *out, cudaStream_t stream, int sm_count) {
    const int64_t nquads = n / 4;
    const int threads = 256;
    int64_t want = (nquads + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count * 8;
    const int grid = (int)(want < cap ? want : cap);
    if (grid <= 0) return QDQ_OK;
    const uint8_t *src = (const uint8_t *)blocks;
    switch (type) {
        case QDQ_Q4_K: dequant_kernel<QDQ_Q4_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q6_K: dequant_kernel<QDQ_Q6_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q8_0: dequant_kernel<QDQ_Q8_0><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q4_0: dequant_kernel<QDQ_Q4_0><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        default: return QDQ_ERR_TYPE;
    }
    return cudaGetLastError() == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

}  // namespace qdq
