// qdq_dequant.cu -- standalone dequantisation: blocks -> fp32, bit-exact.
//
// "S21 The Capstone: picoLM, in Python", section 2 (dequantize_q4_K: raw blocks
// and a count n in, n floats out); "PicoLM Q6_K quantisation bug"
// (dequantize_row_q6_K with the is + l/16 scale index); "PETIT" (q8_0, q4_0).
//
// Also the further GGUF formats (Q5_0, Q5_1, ggml q8_0, Q2_K, Q5_K, Q3_K; ggml
// block layouts).
//
// One thread produces 4 consecutive weights and writes them with one 16-byte
// store, so a warp writes 512 contiguous bytes per instruction. The kernel is
// bound by the fp32 write (4 bytes out per 0.56-1.13 bytes in).
#include <cstdint>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {

template <int TYPE>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ blocks, int64_t nquads,
                                                      float *__restrict__ out) {
    constexpr int kQuads = fmt_weights(TYPE) / 4;  // quads per block
    constexpr int kBytes = fmt_bytes(TYPE);
    // A warp takes 64 consecutive quads: lane l decodes quads l and l + 32 (two
    // independent decodes in flight per thread; each store instruction of the warp
    // still writes 512 contiguous bytes).
    const int lane = threadIdx.x & 31;
    const int64_t nspans = (nquads + 63) / 64;
    const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < nspans; w += wstride) {
        const int64_t t0 = 64 * w + lane, t1 = t0 + 32;
        const int64_t b0 = t0 / kQuads, b1 = t1 / kQuads;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (t0 < nquads) v0 = decode4<TYPE>(blocks + b0 * kBytes, (int)(t0 - b0 * kQuads) * 4);
        if (t1 < nquads) v1 = decode4<TYPE>(blocks + b1 * kBytes, (int)(t1 - b1 * kQuads) * 4);
        if (t0 < nquads) reinterpret_cast<float4 *>(out)[t0] = v0;
        if (t1 < nquads) reinterpret_cast<float4 *>(out)[t1] = v1;
    }
}

int launch_dequant(int type, const void *blocks, int64_t n, float *out, cudaStream_t stream, int sm_count) {
    const int64_t nquads = n / 4;
    const int threads = 256;
    int64_t want = (nquads / 2 + threads - 1) / threads;  // two quads per thread
    const int64_t cap = (int64_t)sm_count * 8;
    const int grid = (int)(want < cap ? want : cap);
    if (grid <= 0) return QDQ_OK;
    const uint8_t *src = (const uint8_t *)blocks;
    switch (type) {
        case QDQ_Q4_K: dequant_kernel<QDQ_Q4_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q6_K: dequant_kernel<QDQ_Q6_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q8_0: dequant_kernel<QDQ_Q8_0><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q4_0: dequant_kernel<QDQ_Q4_0><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q5_0: dequant_kernel<QDQ_Q5_0><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q5_1: dequant_kernel<QDQ_Q5_1><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q8_0_GGML: dequant_kernel<QDQ_Q8_0_GGML><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q2_K: dequant_kernel<QDQ_Q2_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q5_K: dequant_kernel<QDQ_Q5_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q3_K: dequant_kernel<QDQ_Q3_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        default: return QDQ_ERR_TYPE;
    }
    return cudaGetLastError() == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

}  // namespace qdq
