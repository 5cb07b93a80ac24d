// qdq_quantize.cu -- the step before the path: fp32 values -> PETIT q8_0 / q4_0
// blocks (the exporter's quantisation), and a reader for the GGUF container's
// header and tensor index.
//
// Quantiser: "PETIT -- a tiny, CPU-first, quantized LLM inference engine", What
// makes it fast & small (q8_0: 32 weights share an fp32 scale, int8 quants;
// q4_0: fp16 scale + 4-bit nibbles, 18 bytes per 32) and How the pieces match
// (fp32 scale followed by 32 int8, zero-padded to a multiple of 32; q4_0 read as
// (q - 8) * d, weights 0..15 in the low nibbles). The scale rule is not on the
// pages; the symmetric reading is d = amax / 127 (q8_0) and d = fp16(amax / 7)
// (q4_0), quants rounded half to even in binary32.
//
// GGUF: "S21 The Capstone: picoLM, in Python", section 1 (a header,
// self-describing metadata, a tensor index of (name, shape, type, offset),
// padding to general.alignment, then one blob; every tensor is a byte range at
// a known offset). The field encodings (little-endian counts, length-prefixed
// strings, value type codes, type ids) follow the published GGUF description.
#include <cstring>

#include <cuda_fp16.h>

#include "qdq_internal.h"

namespace qdq {
namespace {

// One warp per block of 32 values (grid-stride over blocks): lane i holds x_i,
// the block's max |x| is a warp reduction, and each lane decides its own quant.
template <int TYPE>
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ x, int64_t n,
                                                       uint8_t *__restrict__ out, int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = w0; b < nblocks; b += nw) {
        const int64_t i = b * 32 + lane;
        const float v = i < n ? __ldcs(x + i) : 0.0f;  // the padding past n is zeros
        float a = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
        if constexpr (TYPE == QDQ_Q8_0) {
            const float d = __fdiv_rn(a, 127.0f);
            const float q = d == 0.0f ? 0.0f : fminf(fmaxf(rintf(__fdiv_rn(v, d)), -127.0f), 127.0f);
            uint8_t *blk = out + b * 36;
            if (lane == 0) *reinterpret_cast<float *>(blk) = d;
            blk[4 + lane] = (uint8_t)(int8_t)(int)q;
        } else {
            const __half d16 = __float2half_rn(__fdiv_rn(a, 7.0f));
            const float d = __half2float(d16);
            const int q = d == 0.0f ? 8 : (int)fminf(fmaxf(rintf(__fdiv_rn(v, d)) + 8.0f, 0.0f), 15.0f);
            const int hi = __shfl_down_sync(0xFFFFFFFFu, q, 16);
            uint8_t *blk = out + b * 18;
            if (lane == 0) *reinterpret_cast<__half *>(blk) = d16;
            if (lane < 16) blk[2 + lane] = (uint8_t)(q | (hi << 4));
        }
    }
}

}  // namespace

int launch_quantize(int type, const float *x, int64_t n, void *blocks, cudaStream_t stream, int sm_count) {
    const int64_t nblocks = (n + 31) / 32;
    if (nblocks == 0) return QDQ_OK;
    const int64_t want = (nblocks + 7) / 8;  // CTAs of eight warps
    const int grid = (int)(want < (int64_t)sm_count * 16 ? want : (int64_t)sm_count * 16);
    if (type == QDQ_Q8_0)
        quantize_kernel<QDQ_Q8_0><<<grid, 256, 0, stream>>>(x, n, (uint8_t *)blocks, nblocks);
    else
        quantize_kernel<QDQ_Q4_0><<<grid, 256, 0, stream>>>(x, n, (uint8_t *)blocks, nblocks);
    return cudaGetLastError() == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// GGUF reader (host). A cursor over the mapped bytes; every read is bounds
// checked, so a truncated or malformed file gives QDQ_ERR_FORMAT.
// ---------------------------------------------------------------------------
namespace {

struct Cursor {
    const uint8_t *p;
    int64_t size, at;
    bool ok = true;
    bool take(void *dst, int64_t n) {
        if (!ok || n < 0 || at + n > size) return ok = false;
        std::memcpy(dst, p + at, (size_t)n);
        at += n;
        return true;
    }
    bool skip(int64_t n) {
        if (!ok || n < 0 || at + n > size) return ok = false;
        at += n;
        return true;
    }
    uint32_t u32() {
        uint32_t v = 0;
        take(&v, 4);
        return v;
    }
    uint64_t u64() {
        uint64_t v = 0;
        take(&v, 8);
        return v;
    }
    // a length-prefixed string: its bytes stay in the file
    bool str(int64_t *off, uint64_t *len) {
        *len = u64();
        *off = at;
        return skip((int64_t)*len) && *len < ((uint64_t)1 << 40);
    }
};

// GGUF metadata value types: 0 u8, 1 i8, 2 u16, 3 i16, 4 u32, 5 i32, 6 f32,
// 7 bool, 8 string, 9 array, 10 u64, 11 i64, 12 f64.
int scalar_size(uint32_t t) {
    switch (t) {
        case 0: case 1: case 7: return 1;
        case 2: case 3: return 2;
        case 4: case 5: case 6: return 4;
        case 10: case 11: case 12: return 8;
        default: return -1;
    }
}

bool skip_value(Cursor &c, uint32_t t, int depth = 0) {
    const int sz = scalar_size(t);
    if (sz > 0) return c.skip(sz);
    if (t == 8) {
        int64_t off;
        uint64_t len;
        return c.str(&off, &len);
    }
    if (t == 9 && depth == 0) {
        const uint32_t et = c.u32();
        const uint64_t count = c.u64();
        if (!c.ok || count > ((uint64_t)1 << 40)) return c.ok = false;
        const int esz = scalar_size(et);
        if (esz > 0) return c.skip((int64_t)count * esz);
        for (uint64_t i = 0; i < count && c.ok; ++i) skip_value(c, et, depth + 1);
        return c.ok;
    }
    return c.ok = false;
}

// Bytes per block and values per block of the ggml tensor types the reader knows.
void ggml_geometry(uint32_t t, int *bb, int *bw, int *qdq_type) {
    *qdq_type = 0;
    switch (t) {
        case 0: *bb = 4, *bw = 1; break;                             // f32
        case 1: *bb = 2, *bw = 1; break;                             // f16
        case 2: *bb = 18, *bw = 32, *qdq_type = QDQ_Q4_0; break;     // q4_0: fp16 d + 16 nibble bytes
        case 3: *bb = 20, *bw = 32; break;                           // q4_1
        case 6: *bb = 22, *bw = 32, *qdq_type = QDQ_Q5_0; break;     // q5_0
        case 7: *bb = 24, *bw = 32, *qdq_type = QDQ_Q5_1; break;     // q5_1
        case 8: *bb = 34, *bw = 32, *qdq_type = QDQ_Q8_0_GGML; break;  // ggml q8_0 (fp16 scale)
        case 10: *bb = 84, *bw = 256, *qdq_type = QDQ_Q2_K; break;   // q2_K
        case 11: *bb = 110, *bw = 256, *qdq_type = QDQ_Q3_K; break;  // q3_K
        case 12: *bb = 144, *bw = 256, *qdq_type = QDQ_Q4_K; break;  // q4_K
        case 13: *bb = 176, *bw = 256, *qdq_type = QDQ_Q5_K; break;  // q5_K
        case 14: *bb = 210, *bw = 256, *qdq_type = QDQ_Q6_K; break;  // q6_K
        default: *bb = 0, *bw = 1; break;
    }
}

}  // namespace
}  // namespace qdq

using namespace qdq;

extern "C" {

int qdq_quantize(int type, const float *x, int64_t n, void *blocks, qdq_stream_t stream) {
    if (type != QDQ_Q8_0 && type != QDQ_Q4_0) return QDQ_ERR_TYPE;
    if (n < 0) return QDQ_ERR_SHAPE;
    if (n == 0) return QDQ_OK;
    int rc = QDQ_OK;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    if (x == nullptr || blocks == nullptr) return QDQ_ERR_PTR;
    if (((uintptr_t)x & 15) || ((uintptr_t)blocks & 15)) return QDQ_ERR_ALIGN;
    return launch_quantize(type, x, n, blocks, (cudaStream_t)stream, dev.sm_count);
}

int qdq_gguf_parse(const void *file, int64_t size, qdq_gguf_tensor *tensors, int max_tensors, int *n_tensors,
                   int64_t *data_offset, uint32_t *alignment) {
    if (file == nullptr || n_tensors == nullptr || (max_tensors > 0 && tensors == nullptr)) return QDQ_ERR_PTR;
    *n_tensors = 0;
    Cursor c{(const uint8_t *)file, size, 0};
    const uint32_t magic = c.u32(), version = c.u32();
    if (!c.ok || magic != 0x46554747u || version < 2 || version > 3) return QDQ_ERR_FORMAT;  // "GGUF"
    const uint64_t nt = c.u64(), nkv = c.u64();
    if (!c.ok || nt > (1u << 24) || nkv > (1u << 24)) return QDQ_ERR_FORMAT;
    uint32_t align = 32;
    for (uint64_t i = 0; i < nkv; ++i) {
        int64_t koff;
        uint64_t klen;
        if (!c.str(&koff, &klen)) return QDQ_ERR_FORMAT;
        const uint32_t t = c.u32();
        if (klen == 17 && std::memcmp(c.p + koff, "general.alignment", 17) == 0 && t == 4) {
            align = c.u32();
            if (!c.ok || align == 0 || (align & (align - 1))) return QDQ_ERR_FORMAT;
        } else if (!skip_value(c, t)) {
            return QDQ_ERR_FORMAT;
        }
    }
    if ((int64_t)nt > max_tensors) return QDQ_ERR_LIMIT;
    for (uint64_t i = 0; i < nt; ++i) {
        qdq_gguf_tensor &T = tensors[i];
        std::memset(&T, 0, sizeof(T));
        int64_t noff;
        uint64_t nlen;
        if (!c.str(&noff, &nlen) || nlen >= sizeof(T.name)) return QDQ_ERR_FORMAT;
        std::memcpy(T.name, c.p + noff, (size_t)nlen);
        T.n_dims = (int32_t)c.u32();
        if (!c.ok || T.n_dims < 1 || T.n_dims > 4) return QDQ_ERR_FORMAT;
        int64_t nel = 1;
        for (int d = 0; d < T.n_dims; ++d) {
            T.dims[d] = (int64_t)c.u64();
            if (T.dims[d] < 0 || T.dims[d] > ((int64_t)1 << 40)) return QDQ_ERR_FORMAT;
            nel *= T.dims[d];
            if (nel > ((int64_t)1 << 42)) return QDQ_ERR_FORMAT;
        }
        T.ggml_type = (int32_t)c.u32();
        T.offset = (int64_t)c.u64();
        if (!c.ok || T.offset < 0 || (T.offset % align)) return QDQ_ERR_FORMAT;
        int bb, bw;
        ggml_geometry((uint32_t)T.ggml_type, &bb, &bw, &T.qdq_type);
        if (bb > 0 && T.dims[0] % bw) return QDQ_ERR_FORMAT;  // rows are whole blocks
        T.bytes = bb > 0 ? nel / bw * bb : 0;
    }
    const int64_t data = (c.at + align - 1) / align * align;
    for (uint64_t i = 0; i < nt; ++i) {  // every known-size tensor inside the file
        tensors[i].offset += data;
        if (tensors[i].offset + tensors[i].bytes > size) return QDQ_ERR_FORMAT;
    }
    *n_tensors = (int)nt;
    if (data_offset) *data_offset = data;
    if (alignment) *alignment = align;
    return QDQ_OK;
}

int qdq_gguf_find_kv(const void *file, int64_t size, const char *key, uint32_t *value_type,
                     int64_t *value_offset) {
    if (file == nullptr || key == nullptr || value_type == nullptr || value_offset == nullptr) return QDQ_ERR_PTR;
    Cursor c{(const uint8_t *)file, size, 0};
    const uint32_t magic = c.u32(), version = c.u32();
    if (!c.ok || magic != 0x46554747u || version < 2 || version > 3) return QDQ_ERR_FORMAT;
    c.u64();
    const uint64_t nkv = c.u64();
    if (!c.ok || nkv > (1u << 24)) return QDQ_ERR_FORMAT;
    const size_t klen_want = std::strlen(key);
    for (uint64_t i = 0; i < nkv; ++i) {
        int64_t koff;
        uint64_t klen;
        if (!c.str(&koff, &klen)) return QDQ_ERR_FORMAT;
        const uint32_t t = c.u32();
        if (!c.ok) return QDQ_ERR_FORMAT;
        if (klen == klen_want && std::memcmp(c.p + koff, key, klen) == 0) {
            *value_type = t;
            *value_offset = c.at;
            return QDQ_OK;
        }
        if (!skip_value(c, t)) return QDQ_ERR_FORMAT;
    }
    return QDQ_ERR_NOT_FOUND;
}

}  // extern "C"
