// qdq_dequant.cu -- standalone dequantisation: blocks -> fp32, bit-exact.
//
// "S21 The Capstone: picoLM, in Python", section 2 (dequantize_q4_K: raw blocks
// and a count n in, n floats out); "PicoLM Q6_K quantisation bug"
// (dequantize_row_q6_K with the is + l/16 scale index); "PETIT" (q8_0, q4_0).
//
// Also the further GGUF formats (Q5_0, Q5_1, ggml q8_0, Q2_K; ggml block layouts).
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
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < nquads; t += stride) {
        const int64_t b = t / kQuads;
        const int e0 = (int)(t - b * kQuads) * 4;
        reinterpret_cast<float4 *>(out)[t] = decode4<TYPE>(blocks + b * kBytes, e0);
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
        case QDQ_Q5_0: dequant_kernel<QDQ_Q5_0><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q5_1: dequant_kernel<QDQ_Q5_1><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q8_0_GGML: dequant_kernel<QDQ_Q8_0_GGML><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        case QDQ_Q2_K: dequant_kernel<QDQ_Q2_K><<<grid, threads, 0, stream>>>(src, nquads, out); break;
        default: return QDQ_ERR_TYPE;
    }
    return cudaGetLastError() == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

}  // namespace qdq
