// qdq_gemv_more.cu -- fused dequant-GEMV for the further GGUF formats (Q5_0,
// Q5_1, ggml q8_0, Q2_K, Q5_K, Q3_K; ggml block layouts, a reading: the pages name these
// formats and give Q2_K's size, "S21 The Capstone: picoLM, in Python", section 2).
//
// y[b][r] = sum_c w[r][c] x[b][c] with each weight decoded by the shared decoder
// (decode4, the same arithmetic as the standalone dequantisation, so every weight
// is the format's exact fp32 value) and multiplied straight into fp32
// accumulators: only the quantised bytes cross the memory bus ("S21", section 3).
// One warp per row (grid-stride over rows); lane i takes the row's quads of four
// weights i, i + 32, ...; each batch column's x is read through the read-only
// cache (every row reads the same x). The warp's lanes add up by shuffles, lane
// 0 stores y. Bound: the decode's issue rate, not HBM: a simpler design than the
// streaming kernel, for formats outside the main four.
#include <cstdint>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {
namespace {

template <int TYPE, int BT>
__global__ void __launch_bounds__(256) gemv_more_kernel(const uint8_t *__restrict__ W, int64_t rows, int64_t cols,
                                                        const float *__restrict__ x, float *__restrict__ y,
                                                        int batch) {
    constexpr int kQuads = fmt_weights(TYPE) / 4, kBytes = fmt_bytes(TYPE);
    const int lane = threadIdx.x & 31;
    const int64_t nq = cols / 4, rb = cols / fmt_weights(TYPE) * kBytes;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = w0; r < rows; r += nw) {
        const uint8_t *row = W + r * rb;
        float acc[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[b] = 0.f;
        for (int64_t qd = lane; qd < nq; qd += 32) {
            const int64_t blk = qd / kQuads;
            const float4 w = decode4<TYPE>(row + blk * kBytes, (int)(qd - blk * kQuads) * 4);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                if (b < batch) {
                    const float4 xv = __ldg(reinterpret_cast<const float4 *>(x + (int64_t)b * cols) + qd);
                    acc[b] = fmaf(w.x, xv.x, acc[b]);
                    acc[b] = fmaf(w.y, xv.y, acc[b]);
                    acc[b] = fmaf(w.z, xv.z, acc[b]);
                    acc[b] = fmaf(w.w, xv.w, acc[b]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], o);
            if (lane == 0 && b < batch) y[(int64_t)b * rows + r] = acc[b];
        }
    }
}

template <int TYPE>
int launch_type(const uint8_t *W, int64_t rows, int64_t cols, const float *x, float *y, int batch, int grid,
                cudaStream_t stream) {
    if (batch <= 1)
        gemv_more_kernel<TYPE, 1><<<grid, 256, 0, stream>>>(W, rows, cols, x, y, batch);
    else if (batch <= 2)
        gemv_more_kernel<TYPE, 2><<<grid, 256, 0, stream>>>(W, rows, cols, x, y, batch);
    else if (batch <= 4)
        gemv_more_kernel<TYPE, 4><<<grid, 256, 0, stream>>>(W, rows, cols, x, y, batch);
    else
        gemv_more_kernel<TYPE, 8><<<grid, 256, 0, stream>>>(W, rows, cols, x, y, batch);
    return cudaGetLastError() == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

}  // namespace

bool is_more_type(int type) {
    return type == QDQ_Q5_0 || type == QDQ_Q5_1 || type == QDQ_Q8_0_GGML || type == QDQ_Q2_K || type == QDQ_Q5_K ||
           type == QDQ_Q3_K;
}

int launch_gemv_more(int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y, int batch,
                     cudaStream_t stream, int sm_count) {
    const int64_t warps_wanted = rows, cap = (int64_t)sm_count * 16;  // CTAs of 8 warps
    const int grid = (int)((warps_wanted + 7) / 8 < cap ? (warps_wanted + 7) / 8 : cap);
    const uint8_t *w = (const uint8_t *)W;
    for (int b0 = 0; b0 < batch; b0 += 8) {  // batch slices of at most 8 columns
        const int nb = batch - b0 < 8 ? batch - b0 : 8;
        const float *xs = x + (int64_t)b0 * cols;
        float *ys = y + (int64_t)b0 * rows;
        int rc;
        switch (type) {
            case QDQ_Q5_0: rc = launch_type<QDQ_Q5_0>(w, rows, cols, xs, ys, nb, grid, stream); break;
            case QDQ_Q5_1: rc = launch_type<QDQ_Q5_1>(w, rows, cols, xs, ys, nb, grid, stream); break;
            case QDQ_Q8_0_GGML: rc = launch_type<QDQ_Q8_0_GGML>(w, rows, cols, xs, ys, nb, grid, stream); break;
            case QDQ_Q2_K: rc = launch_type<QDQ_Q2_K>(w, rows, cols, xs, ys, nb, grid, stream); break;
            case QDQ_Q5_K: rc = launch_type<QDQ_Q5_K>(w, rows, cols, xs, ys, nb, grid, stream); break;
            case QDQ_Q3_K: rc = launch_type<QDQ_Q3_K>(w, rows, cols, xs, ys, nb, grid, stream); break;
            default: return QDQ_ERR_TYPE;
        }
        if (rc) return rc;
    }
    return QDQ_OK;
}

}  // namespace qdq
