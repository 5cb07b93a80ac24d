// qdq_llama.cu -- the decode-step glue around the GEMV plans: the attention block
// of one position (RoPE, fp16 key/value cache, GQA attention with an online
// softmax) and a one-token forward pass of a Llama-architecture model built from
// plans whose GEMVs carry the rmsnorm, SwiGLU, residual and argmax options.
//
// "S21 The Capstone: picoLM, in Python", section 4 (model_forward(m, token, pos):
// the embedding row, per layer rmsnorm -> q/k/v -> rope -> fp16 cache at pos ->
// per-head attention with an online softmax and GQA -> output projection ->
// SwiGLU -> residuals; final rmsnorm and output matmul) and section 3 (the
// interleaved RoPE layout: pairs (x[2i], x[2i+1])); "PETIT", How the pieces match
// (RoPE base 10000, applied per head).
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_fp16.h>

#include "qdq_internal.h"

namespace qdq {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxHeadDim = 256;

// Pair frequencies base^(-2i / head_dim), computed on the host in double.
struct RopeFreqs {
    double f[kMaxHeadDim / 2];
};

// One CTA per query head h (KV head g = h / kv_mul).
//  1. Angles: pos * f_i reaches thousands of radians, where a float angle would
//     be off by 1e-4. The product and its reduction by 2 pi are formed in double
//     (four double operations: the frequencies come from the host, as double
//     transcendentals are slow on this GPU), then sincosf of the reduced angle.
//  2. q_h and k_g turn pair by pair; k and v are rounded to fp16 (the cache is
//     fp16), and the first query head of the group stores them at position pos.
//  3. Online softmax over t <= pos in chunks of 32 positions: warp w takes chunks
//     w, w + 8, ...; each keeps a running maximum m, sum l and weighted value
//     sum, rescaled when m grows; the warps' states are merged at the end. No
//     score array exists. The current position's key and value come from shared
//     memory (their fp16 values), so no CTA reads a cache entry another CTA is
//     writing.
__global__ void __launch_bounds__(kAttnThreads) rope_attn_kernel(const float *__restrict__ q, const float *__restrict__ k,
                                                                 const float *__restrict__ v, __half *k_cache,
                                                                 __half *v_cache, float *__restrict__ out,
                                                                 int n_heads, int n_kv_heads, int D, int pos,
                                                                 const __grid_constant__ RopeFreqs fr) {
    __shared__ float qs[kMaxHeadDim], kc[kMaxHeadDim], vc[kMaxHeadDim];
    __shared__ float wm[kAttnWarps], wl[kAttnWarps];
    __shared__ float wacc[kAttnWarps][kMaxHeadDim];
    const int h = blockIdx.x, kv_mul = n_heads / n_kv_heads, g = h / kv_mul;
    const int kvd = n_kv_heads * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool writer = (h % kv_mul) == 0;

    for (int i = tid; i < D / 2; i += kAttnThreads) {
        const double th = (double)pos * fr.f[i];
        const double kq = rint(th * 0.15915494309189535);  // turns: th / (2 pi)
        const float r = (float)fma(-kq, 6.283185307179586, th);
        float s, c;
        __sincosf(r, &s, &c);  // |r| <= pi: the fast form is accurate to ~4e-7
        const float qa = q[h * D + 2 * i], qb = q[h * D + 2 * i + 1];
        qs[2 * i] = qa * c - qb * s;
        qs[2 * i + 1] = qa * s + qb * c;
        const float ka = k[g * D + 2 * i], kb = k[g * D + 2 * i + 1];
        const __half k0 = __float2half_rn(ka * c - kb * s), k1 = __float2half_rn(ka * s + kb * c);
        const __half v0 = __float2half_rn(v[g * D + 2 * i]), v1 = __float2half_rn(v[g * D + 2 * i + 1]);
        kc[2 * i] = __half2float(k0);
        kc[2 * i + 1] = __half2float(k1);
        vc[2 * i] = __half2float(v0);
        vc[2 * i + 1] = __half2float(v1);
        if (writer) {
            const int64_t o = (int64_t)pos * kvd + g * D + 2 * i;
            k_cache[o] = k0;
            k_cache[o + 1] = k1;
            v_cache[o] = v0;
            v_cache[o + 1] = v1;
        }
    }
    __syncthreads();

    const float inv = 1.0f / sqrtf((float)D);
    constexpr int kPer2 = kMaxHeadDim / 64;  // dim pairs per lane in the value sums
    constexpr int kPer = 2 * kPer2;          // acc[2 j], acc[2 j + 1]: dims 2 (lane + 32 j), + 1
    float m = -INFINITY, l = 0.f, acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    const bool vec = (D & 7) == 0;  // key rows as 16-byte loads
    // Warp w takes the 32-position chunks w, w + 8, ...: lane i scores position
    // c0 + i over the whole head (its row's loads independent of the other
    // lanes'), the chunk's maximum and weights come from warp reductions, then
    // the lanes switch to dims and add the chunk's weighted values.
    for (int c0 = 32 * warp; c0 <= pos; c0 += 32 * kAttnWarps) {
        const int t = c0 + lane;
        float s = -INFINITY;
        if (t <= pos) {
            float dot = 0.f;
            if (t == pos) {
                for (int d = 0; d < D; ++d) dot += qs[d] * kc[d];
            } else if (vec) {
                const uint4 *kr = reinterpret_cast<const uint4 *>(k_cache + (int64_t)t * kvd + g * D);
                for (int e = 0; e < D / 8; ++e) {
                    const uint4 u = kr[e];
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(h2[i]);
                        dot += qs[8 * e + 2 * i] * f.x + qs[8 * e + 2 * i + 1] * f.y;
                    }
                }
            } else {
                const __half *kr = k_cache + (int64_t)t * kvd + g * D;
                for (int d = 0; d < D; ++d) dot += qs[d] * __half2float(kr[d]);
            }
            s = dot * inv;
        }
        float cm = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
        const float mn = fmaxf(m, cm);
        const float scale = expf(m - mn);  // 0 for the first chunk (m = -inf)
        const float p = t <= pos ? expf(s - mn) : 0.f;
        float ps = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, o);
        l = l * scale + ps;
#pragma unroll
        for (int j = 0; j < kPer; ++j) acc[j] *= scale;
        // weighted values: lane holds the dim pairs 2 lane + 64 j; positions before
        // pos from the cache (independent loads), pos itself from shared memory
        const int last = pos - c0 < 31 ? pos - c0 : 31;  // the chunk's last position, relative
        const int nh = c0 + last == pos ? last : last + 1;  // ... of them in the cache
        const __half2 *vrow = reinterpret_cast<const __half2 *>(v_cache + (int64_t)c0 * kvd + g * D);
#pragma unroll 8
        for (int u = 0; u < nh; ++u) {
            const float pu = __shfl_sync(0xFFFFFFFFu, p, u);
#pragma unroll
            for (int j = 0; j < kPer2; ++j) {
                const int d2 = lane + 32 * j;  // pair index
                if (2 * d2 < D) {
                    const float2 f = __half22float2(vrow[(int64_t)u * (kvd / 2) + d2]);
                    acc[2 * j] += pu * f.x;
                    acc[2 * j + 1] += pu * f.y;
                }
            }
        }
        if (nh <= last) {  // pos is in this chunk
            const float pu = __shfl_sync(0xFFFFFFFFu, p, last);
#pragma unroll
            for (int j = 0; j < kPer2; ++j) {
                const int d2 = lane + 32 * j;
                if (2 * d2 < D) {
                    acc[2 * j] += pu * vc[2 * d2];
                    acc[2 * j + 1] += pu * vc[2 * d2 + 1];
                }
            }
        }
        m = mn;
    }
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
#pragma unroll
    for (int j = 0; j < kPer2; ++j) {
        const int d2 = lane + 32 * j;
        if (2 * d2 < D) {
            wacc[warp][2 * d2] = acc[2 * j];
            wacc[warp][2 * d2 + 1] = acc[2 * j + 1];
        }
    }
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w]);
    float L = 0.f;
    for (int w = 0; w < kAttnWarps; ++w)
        if (wl[w] > 0.f) L += wl[w] * expf(wm[w] - M);
    for (int d = tid; d < D; d += kAttnThreads) {
        float o = 0.f;
        for (int w = 0; w < kAttnWarps; ++w)
            if (wl[w] > 0.f) o += wacc[w][d] * expf(wm[w] - M);
        out[h * D + d] = o / L;
    }
}

}  // namespace

int launch_rope_attention(const float *q, const float *k, const float *v, uint16_t *k_cache, uint16_t *v_cache,
                          float *out, int n_heads, int n_kv_heads, int head_dim, int pos, float rope_base,
                          cudaStream_t stream) {
    RopeFreqs fr;
    for (int i = 0; i < head_dim / 2; ++i) fr.f[i] = std::pow((double)rope_base, -2.0 * i / (double)head_dim);
    rope_attn_kernel<<<n_heads, kAttnThreads, 0, stream>>>(q, k, v, (__half *)k_cache, (__half *)v_cache, out,
                                                           n_heads, n_kv_heads, head_dim, pos, fr);
    if (cudaGetLastError() != cudaSuccess) return QDQ_ERR_CUDA;
    return QDQ_OK;
}

}  // namespace qdq

using namespace qdq;

// A model instance: the caller's weights, the library's activations, fp16 cache
// and plans. Buffers in one device allocation:
//   h[dim] (residual stream), q[dim], k[kv], v[kv], att[dim], gate[hidden],
//   up[hidden], logits[vocab], argmax (int64), then the key and value caches
//   [n_layers][max_seq][kv] fp16.
struct qdq_llama {
    qdq_llama_config cfg{};
    int device = -1;
    const void *embd = nullptr;
    int embd_type = 0;
    int64_t embd_row_bytes = 0;
    char *mem = nullptr;
    float *h = nullptr, *q = nullptr, *k = nullptr, *v = nullptr, *att = nullptr, *gate = nullptr, *up = nullptr,
          *logits = nullptr;
    int64_t *argmax = nullptr;
    uint16_t *kcache = nullptr, *vcache = nullptr;
    qdq_plan *plan = nullptr;  // every layer and the head, attention levels included
};

namespace {

int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

int check_config(const qdq_llama_config *c) {
    if (c->dim < 1 || c->hidden < 1 || c->n_layers < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->vocab < 1 ||
        c->max_seq < 1)
        return QDQ_ERR_SHAPE;
    if (c->dim % c->n_heads || c->n_heads % c->n_kv_heads) return QDQ_ERR_SHAPE;
    const int D = c->dim / c->n_heads;
    if (D % 2 || D > kMaxHeadDim) return QDQ_ERR_SHAPE;
    if (!(c->rope_base > 1.0f) || !(c->norm_eps >= 0.0f)) return QDQ_ERR_SHAPE;
    if (c->n_layers > 1024 || c->vocab > (1 << 30) || c->max_seq > (1 << 24)) return QDQ_ERR_LIMIT;
    return QDQ_OK;
}

}  // namespace

extern "C" {

int qdq_rope_attention(const float *q, const float *k, const float *v, uint16_t *k_cache, uint16_t *v_cache,
                       float *out, int n_heads, int n_kv_heads, int head_dim, int pos, int max_seq, float rope_base,
                       qdq_stream_t stream) {
    if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim < 2 || head_dim % 2 ||
        head_dim > kMaxHeadDim || pos < 0 || pos >= max_seq || !(rope_base > 1.0f))
        return QDQ_ERR_SHAPE;
    if (!q || !k || !v || !k_cache || !v_cache || !out) return QDQ_ERR_PTR;
    int rc = QDQ_OK;
    current_device(&rc);
    if (rc) return rc;
    return launch_rope_attention(q, k, v, k_cache, v_cache, out, n_heads, n_kv_heads, head_dim, pos, rope_base,
                                 (cudaStream_t)stream);
}

int qdq_llama_create(const qdq_llama_config *cfg, const void *token_embd, int embd_type,
                     const qdq_llama_layer *layers, const float *output_norm, const void *output, int output_type,
                     qdq_llama **out) {
    if (out == nullptr || cfg == nullptr || layers == nullptr || token_embd == nullptr || output_norm == nullptr ||
        output == nullptr)
        return QDQ_ERR_PTR;
    *out = nullptr;
    int rc = check_config(cfg);
    if (rc) return rc;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    if (qdq_block_weights(embd_type) <= 0 || qdq_block_weights(output_type) <= 0) return QDQ_ERR_TYPE;
    if (cfg->dim % qdq_block_weights(embd_type)) return QDQ_ERR_SHAPE;
    // the embedding row is decoded in place: its first byte must be 16-byte aligned
    if (((int64_t)cfg->dim / qdq_block_weights(embd_type) * qdq_block_bytes(embd_type)) % 16) return QDQ_ERR_ALIGN;
    qdq_llama *m = new (std::nothrow) qdq_llama();
    if (!m) return QDQ_ERR_CUDA;
    m->cfg = *cfg;
    m->device = dev.device;
    m->embd = token_embd;
    m->embd_type = embd_type;
    m->embd_row_bytes = (int64_t)cfg->dim / qdq_block_weights(embd_type) * qdq_block_bytes(embd_type);
    const int64_t dim = cfg->dim, hid = cfg->hidden, kv = (int64_t)cfg->n_kv_heads * (cfg->dim / cfg->n_heads);
    const int64_t cache = (int64_t)cfg->n_layers * cfg->max_seq * kv * 2;
    int64_t off[11], total = 0;
    const int64_t sizes[11] = {4 * dim, 4 * dim, 4 * kv, 4 * kv, 4 * dim, 4 * hid, 4 * hid, 4 * (int64_t)cfg->vocab,
                               8, cache, cache};
    for (int i = 0; i < 11; ++i) {
        off[i] = total;
        total += align256(sizes[i]);
    }
    if (cudaMalloc((void **)&m->mem, total) != cudaSuccess || cudaMemset(m->mem, 0, total) != cudaSuccess) {
        cudaGetLastError();
        if (m->mem) cudaFree(m->mem);
        delete m;
        return QDQ_ERR_CUDA;
    }
    m->h = (float *)(m->mem + off[0]);
    m->q = (float *)(m->mem + off[1]);
    m->k = (float *)(m->mem + off[2]);
    m->v = (float *)(m->mem + off[3]);
    m->att = (float *)(m->mem + off[4]);
    m->gate = (float *)(m->mem + off[5]);
    m->up = (float *)(m->mem + off[6]);
    m->logits = (float *)(m->mem + off[7]);
    m->argmax = (int64_t *)(m->mem + off[8]);
    m->kcache = (uint16_t *)(m->mem + off[9]);
    m->vcache = (uint16_t *)(m->mem + off[10]);

    const float eps = cfg->norm_eps;
    auto desc = [](int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y) {
        qdq_gemv_desc d;
        std::memset(&d, 0, sizeof(d));
        d.type = type;
        d.W = W;
        d.rows = rows;
        d.cols = cols;
        d.x = x;
        d.y = y;
        return d;
    };
    auto opt = [](int x_op, int y_op, const float *x2, const float *nw, float e, int64_t *am) {
        qdq_gemv_opts o;
        std::memset(&o, 0, sizeof(o));
        o.x_op = x_op;
        o.y_op = y_op;
        o.x2 = x2;
        o.norm_w = nw;
        o.eps = e;
        o.argmax = am;
        return o;
    };
    std::vector<qdq_gemv_desc> D;
    std::vector<qdq_gemv_opts> O;
    std::vector<int> Lv;
    int level = 0;
    const int D_h = cfg->dim / cfg->n_heads;
    for (int l = 0; l < cfg->n_layers; ++l) {
        const qdq_llama_layer &w = layers[l];
        // q, k, v read rmsnorm(h, attn_norm) (one staged x for the three)
        D.push_back(desc(w.type[0], w.w[0], dim, dim, m->h, m->q));
        D.push_back(desc(w.type[1], w.w[1], kv, dim, m->h, m->k));
        D.push_back(desc(w.type[2], w.w[2], kv, dim, m->h, m->v));
        for (int i = 0; i < 3; ++i) {
            O.push_back(opt(QDQ_X_RMSNORM, QDQ_Y_STORE, nullptr, w.attn_norm, eps, nullptr));
            Lv.push_back(level);
        }
        ++level;
        // attention of this layer: its own level (see kPlanAttnType for the packing)
        qdq_gemv_desc a = desc(kPlanAttnType, m->kcache + (int64_t)l * cfg->max_seq * kv, cfg->n_heads, D_h, m->q,
                               m->att);
        qdq_gemv_opts ao = opt(QDQ_X_PLAIN, QDQ_Y_STORE, m->k, m->v, cfg->rope_base,
                               (int64_t *)(m->vcache + (int64_t)l * cfg->max_seq * kv));
        ao.reserved = cfg->n_kv_heads;
        D.push_back(a);
        O.push_back(ao);
        Lv.push_back(level++);
        // h += Wo att; gate, up from rmsnorm(h, ffn_norm); h += Wdown (silu(gate) * up)
        D.push_back(desc(w.type[3], w.w[3], dim, dim, m->att, m->h));
        O.push_back(opt(QDQ_X_PLAIN, QDQ_Y_ADD, nullptr, nullptr, 0.f, nullptr));
        Lv.push_back(level++);
        // (up to 4096 columns silu is applied once, as the gate is stored, and the
        // down projection stages the product; wider, it stages silu(gate) * up)
        const bool silu_at_store = dim <= 4096;
        D.push_back(desc(w.type[4], w.w[4], hid, dim, m->h, m->gate));
        D.push_back(desc(w.type[5], w.w[5], hid, dim, m->h, m->up));
        O.push_back(opt(QDQ_X_RMSNORM, silu_at_store ? QDQ_Y_SILU : QDQ_Y_STORE, nullptr, w.ffn_norm, eps, nullptr));
        O.push_back(opt(QDQ_X_RMSNORM, QDQ_Y_STORE, nullptr, w.ffn_norm, eps, nullptr));
        Lv.push_back(level);
        Lv.push_back(level);
        ++level;
        D.push_back(desc(w.type[6], w.w[6], dim, hid, m->gate, m->h));
        O.push_back(opt(silu_at_store ? QDQ_X_MUL : QDQ_X_SWIGLU, QDQ_Y_ADD, m->up, nullptr, 0.f, nullptr));
        Lv.push_back(level++);
    }
    // logits = Wout rmsnorm(h, output_norm), with their argmax
    D.push_back(desc(output_type, output, cfg->vocab, dim, m->h, m->logits));
    O.push_back(opt(QDQ_X_RMSNORM, QDQ_Y_STORE, nullptr, output_norm, eps, m->argmax));
    Lv.push_back(level);
    rc = (int)D.size() > kMaxPlanDescs || level + 1 > kMaxPlanLevels
             ? QDQ_ERR_LIMIT
             : plan_create_with_attention(D.data(), O.data(), Lv.data(), (int)D.size(), &m->plan);
    if (rc) {
        qdq_llama_destroy(m);
        return rc;
    }
    *out = m;
    return QDQ_OK;
}

int qdq_llama_forward(qdq_llama *m, int token, int pos, qdq_stream_t stream) {
    if (m == nullptr) return QDQ_ERR_PTR;
    if (token < 0 || token >= m->cfg.vocab || pos < 0 || pos >= m->cfg.max_seq) return QDQ_ERR_SHAPE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != m->device) return QDQ_ERR_DEVICE;
    const qdq_llama_config &c = m->cfg;
    // x = the token's embedding row, decoded; then every layer and the head in one launch
    int rc = qdq_dequant_async(m->embd_type, (const char *)m->embd + (int64_t)token * m->embd_row_bytes, c.dim, m->h,
                               stream);
    if (!rc) rc = plan_set_pos(m->plan, pos);
    if (!rc) rc = qdq_plan_run(m->plan, stream);
    return rc;
}

int qdq_llama_buffers(const qdq_llama *m, float **logits, int64_t **argmax, float **hidden, uint16_t **k_cache,
                      uint16_t **v_cache) {
    if (m == nullptr) return QDQ_ERR_PTR;
    if (logits) *logits = m->logits;
    if (argmax) *argmax = m->argmax;
    if (hidden) *hidden = m->h;
    if (k_cache) *k_cache = m->kcache;
    if (v_cache) *v_cache = m->vcache;
    return QDQ_OK;
}

int qdq_llama_launches(const qdq_llama *m) { return m ? 2 : 0; }

void qdq_llama_destroy(qdq_llama *m) {
    if (m == nullptr) return;
    if (m->plan) qdq_plan_destroy(m->plan);
    if (m->mem) cudaFree(m->mem);
    delete m;
}

}  // extern "C"
