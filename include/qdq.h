/*
 * qdq.h -- C ABI of libqdq: dequantisation and fused dequant-GEMV over
 * block-quantised weights, in hand-written CUDA for sm_103a (GB300).
 *
 * Block formats (all little-endian, see the per-type notes below):
 *   QDQ_Q4_K  GGUF Q4_K, 144 bytes per 256 weights ("S21 The Capstone: picoLM,
 *             in Python", section 2 K-quants): fp16 d, fp16 dmin, 12 bytes of
 *             packed 6-bit scales and mins (one pair per 32-weight sub-block),
 *             128 nibble bytes. w = d*sc*q - dmin*mn.
 *   QDQ_Q6_K  GGUF Q6_K, 210 bytes per 256 weights ("PicoLM Q6_K quantisation
 *             bug", block_q6_K struct): ql[128] low 4 bits, qh[64] high 2 bits,
 *             int8 scales[16] (one per 16 weights), fp16 d. w = d*sc*(q6-32).
 *             The ql/qh bit placement follows the ggml layout.
 *   QDQ_Q8_0  PETIT q8_0, 36 bytes per 32 weights ("PETIT", How the pieces
 *             match): fp32 scale d, 32 int8 q. w = d*q. (Not ggml's q8_0, whose
 *             scale is fp16.)
 *   QDQ_Q4_0  PETIT q4_0, 18 bytes per 32 weights (same section): fp16 scale d,
 *             16 bytes; byte i holds weight i (low nibble) and weight i+16 (high
 *             nibble). w = (q-8)*d.
 *   More GGUF formats. The pages name eight GGUF formats and give Q2_K's size
 *   (84 bytes per 256 weights, "S21 The Capstone: picoLM, in Python", section
 *   2); the layouts follow the published ggml block layouts:
 *   QDQ_Q5_0       22 bytes per 32: fp16 d; qh (4 bytes, little-endian word, bit
 *                  i = fifth bit of weight i); 16 nibble bytes as q4_0.
 *                  w = (q-16)*d, q = nibble | bit << 4.
 *   QDQ_Q5_1       24 bytes per 32: fp16 d, fp16 m, qh, 16 nibble bytes.
 *                  w = q*d + m.
 *   QDQ_Q8_0_GGML  34 bytes per 32: fp16 d, 32 int8. w = q*d.
 *   QDQ_Q2_K       84 bytes per 256: 16 bytes of (scale | min << 4) per 16
 *                  weights, 64 bytes of 2-bit quants (weight 128n + 32j + l: bits
 *                  2j..2j+1 of byte 32n + l, pair 8n + 2j + l/16), fp16 d, fp16
 *                  dmin. w = d*sc*q - dmin*mn.
 *   QDQ_Q5_K       176 bytes per 256: fp16 d, fp16 dmin, the 12 scale/min bytes
 *                  of Q4_K (same packing), qh[32], qs[128]. Weight 64c + 32h + l:
 *                  low four bits in the low (h = 0) or high (h = 1) nibble of
 *                  qs[32c + l], fifth bit at bit 2c + h of qh[l]; sub-block 2c + h.
 *                  w = d*sc*q - dmin*mn, q in 0..31.
 *   QDQ_Q3_K       110 bytes per 256: hmask[32], qs[64], 12 bytes of sixteen
 *                  6-bit scales, fp16 d. Weight 128n + 32j + l: bits 2j..2j+1 of
 *                  qs[32n + l], minus 4 unless bit 4n + j of hmask[l] is set;
 *                  scale s = 8n + 2j + l/16 keeps its low four bits in byte s
 *                  (s < 8, low nibble) or s - 8 (high nibble), its top two at
 *                  bit 2(s/4) of byte 8 + s%4. w = d*(scale - 32)*q.
 *   These six are decoded by qdq_dequant and multiplied by qdq_gemv (a
 *   separate exact-per-weight kernel, any batch); groups and plans take the
 *   main four only (QDQ_ERR_TYPE).
 *
 * Conventions for every call:
 *   - Pointers named W, blocks, x, y, out are DEVICE pointers (cudaMalloc'd or
 *     managed) on the current device, 16-byte aligned. A host pointer gives
 *     QDQ_ERR_PTR, a misaligned one QDQ_ERR_ALIGN, a NULL one QDQ_ERR_PTR.
 *   - A weight matrix is rows x cols (out x in, "PETIT": weights stored out x in,
 *     a projection is one gemv), row-major, each row cols/QK whole blocks.
 *     cols must be a multiple of the block's weight count QK (the caller pads,
 *     as PETIT's exporter does), else QDQ_ERR_SHAPE.
 *   - x is [batch][cols] fp32 and y is [batch][rows] fp32, both contiguous. y is
 *     overwritten, never accumulated into.
 *   - rows == 0 or n == 0 is a no-op returning QDQ_OK.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream). Launch
 *     failures return QDQ_ERR_CUDA. A device-side failure (a bounded wait that
 *     ran out) is recorded in a per-device status word, read back by
 *     qdq_get_device_status(). Nothing aborts, traps or exits.
 *   - The caller owns every buffer. Besides plans (below), the library keeps no
 *     device allocations: only a status word in module memory per device.
 *   - Calls on different streams may run concurrently. Only sm_103 (GB300)
 *     devices are accepted; others give QDQ_ERR_DEVICE.
 */
#ifndef QDQ_H
#define QDQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qdq_stream_t; /* == cudaStream_t */

enum qdq_type {
    QDQ_Q4_0 = 1, QDQ_Q8_0 = 2, QDQ_Q4_K = 3, QDQ_Q6_K = 4,
    /* More GGUF formats (see the notes below the main four): */
    QDQ_Q5_0 = 5, QDQ_Q5_1 = 6, QDQ_Q8_0_GGML = 7, QDQ_Q2_K = 8, QDQ_Q5_K = 9, QDQ_Q3_K = 10
};

enum qdq_status {
    QDQ_OK = 0,
    QDQ_ERR_TYPE = -1,     /* unknown block type */
    QDQ_ERR_SHAPE = -2,    /* negative size, cols or n not a multiple of QK, batch < 1, row too wide */
    QDQ_ERR_ALIGN = -3,    /* a pointer not 16-byte aligned */
    QDQ_ERR_PTR = -4,      /* NULL or host pointer */
    QDQ_ERR_CUDA = -5,     /* a CUDA runtime call or kernel launch failed */
    QDQ_ERR_TIMEOUT = -6,  /* a device-side bounded wait ran out (from qdq_get_device_status) */
    QDQ_ERR_DEVICE = -7,   /* current device is not sm_103 */
    QDQ_ERR_LIMIT = -8,    /* more GEMVs or levels than a plan supports */
    QDQ_ERR_FORMAT = -9,   /* a malformed or truncated GGUF file */
    QDQ_ERR_NOT_FOUND = -10, /* no such GGUF metadata key */
    QDQ_ERR_BOUNDS = -11     /* debug builds (-DQDQ_DEBUG) only: a device-side index or
                                alignment check failed and the access was skipped
                                (from qdq_get_device_status) */
};

/* Bytes per block and weights per block of a type; -1 for an unknown type. */
int qdq_block_bytes(int type);
int qdq_block_weights(int type);

/* Static text for a status code. */
const char *qdq_status_string(int status);

/* ---------------------------------------------------------------------------
 * qdq_dequant: out[i] = w_i for i < n, the fp32 value of each weight.
 * Cited: "S21 The Capstone: picoLM, in Python", section 2 (dequantize_q4_K:
 * raw blocks + count n -> n floats); "PicoLM Q6_K quantisation bug"
 * (dequantize_row_q6_K); "PETIT", What makes it fast & small.
 * `blocks` holds n/QK consecutive blocks; `out` holds n floats. Each value is
 * evaluated in the pages' order with IEEE fp32 round-to-nearest and no fused
 * multiply-add, so the result is bit-for-bit that of a plain CPU decoder.
 * n must be a multiple of QK (QDQ_ERR_SHAPE).
 * qdq_dequant runs on the legacy default stream, qdq_dequant_async on `stream`.
 * ------------------------------------------------------------------------- */
int qdq_dequant(int type, const void *blocks, int64_t n, float *out_f32);
int qdq_dequant_async(int type, const void *blocks, int64_t n, float *out_f32,
                      qdq_stream_t stream);

/* ---------------------------------------------------------------------------
 * qdq_gemv: y[b][r] = sum_c w[r][c] * x[b][c] for b < batch, r < rows,
 * with dequantisation fused into the dot product: only the quantised bytes of W
 * cross the memory bus ("S21 The Capstone: picoLM, in Python", section 3,
 * fused dequant + dot; picoLM's matmul(out, x, W, n, d, type); PETIT gemv_q8 /
 * gemv_q4 / gemm).
 * Accumulation is fp32. Against the exact (double) sum y_ref the result meets
 * |y - y_ref| <= 1e-5 * sum_c |w[r][c] x[b][c]| + 1e-7 for finite inputs.
 * Batch 1..4 (1..3 for q8_0 and q4_0) runs the streaming
 * CUDA-core kernel (each decoded weight meets every batch column); larger
 * batches the tensor-core path (exact integer quants x bf16-split x on tcgen05,
 * scales applied per group in fp32). Any row width is accepted (wide rows are
 * split into column chunks inside the streaming kernel). Neither path allocates
 * memory: the tensor-core kernel splits x into its bf16 operand in shared memory.
 * ------------------------------------------------------------------------- */
int qdq_gemv(int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y,
             int batch, qdq_stream_t stream);

/* One GEMV of a group or plan. */
typedef struct qdq_gemv_desc {
    int32_t type;
    int32_t reserved;
    const void *W;
    int64_t rows;
    int64_t cols;
    const float *x; /* [batch][cols] */
    float *y;       /* [batch][rows] */
} qdq_gemv_desc;

/* Up to 8 independent GEMVs with a common batch, in one launch (for instance
 * q, k and v of one layer, which may mix Q4_K and Q6_K). Same rules as
 * qdq_gemv for each; batch must be <= 8. */
int qdq_gemv_group(const qdq_gemv_desc *descs, int n, int batch, qdq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Plans: a whole decode step's GEMVs in one persistent launch.
 * ("S21 The Capstone: picoLM, in Python", section 4: model_forward runs, per
 * layer, the q/k/v, output, gate/up and down projections, then the output head.)
 * descs[i] belongs to dependency level level[i]; levels must be non-decreasing
 * from 0. All GEMVs of level k complete (their y written and visible) before any
 * GEMV of level k+1 reads its x; weight bytes of later levels may be fetched
 * earlier, since weights never depend on earlier outputs. batch <= 8; at most
 * 192 GEMVs and 128 levels (QDQ_ERR_LIMIT). The plan copies the descriptors
 * (not the buffers they point to, which must stay valid while the plan is run)
 * and allocates one small device array of level counters; destroy frees it.
 * Runs of one plan must not overlap on the GPU. If qdq_get_device_status()
 * reports QDQ_ERR_TIMEOUT after a run, call qdq_plan_reset() before the next.
 * ------------------------------------------------------------------------- */
typedef struct qdq_plan qdq_plan;
int qdq_plan_create(const qdq_gemv_desc *descs, const int *level, int n, int batch,
                    qdq_plan **plan_out);

/* ---------------------------------------------------------------------------
 * Step glue fused into a plan's GEMVs ("S21 The Capstone: picoLM, in Python",
 * section 4, model_forward: rmsnorm before the q/k/v and gate/up projections,
 * SwiGLU between gate/up and down, residual additions after the output and down
 * projections, and the output head whose largest logit greedy decoding takes;
 * "PETIT", What makes it fast & small: RMSNorm + SwiGLU Llama block).
 * opts[i] applies to descs[i]:
 *   x_op  QDQ_X_PLAIN    the GEMV reads x as given.
 *         QDQ_X_RMSNORM  it reads x / sqrt(mean(x^2) + eps) * norm_w (the mean
 *                        over the cols entries of each batch column), computed
 *                        while x is staged; norm_w is [cols] fp32.
 *         QDQ_X_SWIGLU   it reads silu(x) * x2 with silu(g) = g / (1 + exp(-g));
 *                        x is the gate output, x2 the up output, both
 *                        [batch][cols].
 *         QDQ_X_MUL      it reads x * x2 elementwise (x2 [cols]; batch 1): with
 *                        a gate GEMV stored through QDQ_Y_SILU, the same SwiGLU
 *                        product with silu evaluated once per element instead
 *                        of once per CTA that stages it.
 *   y_op  QDQ_Y_STORE    y = W x' (as qdq_gemv).
 *         QDQ_Y_ADD      y += W x' (a residual addition; y must not be read by
 *                        another GEMV of the same level).
 *         QDQ_Y_SILU     y = silu(W x'), the same silu as QDQ_X_SWIGLU's. Batch
 *                        1 and cols <= 4096 (a row's sum is complete in one
 *                        store).
 *   argmax  NULL, or a device int64: after the run it holds the index of the
 *           largest y of this GEMV (the smallest such index on ties). At most
 *           one GEMV of a plan, in its last level, batch 1, cols <= 8192.
 * GEMVs of one level that read the same x must use the same x_op, x2, norm_w
 * and eps. Every option is applied inside the plan's single kernel: no pass of
 * its own. Errors: QDQ_ERR_SHAPE for a rule above broken, QDQ_ERR_PTR /
 * QDQ_ERR_ALIGN for a bad x2, norm_w or argmax pointer. The plan then also
 * owns 16 bytes of device memory for the argmax.
 * ------------------------------------------------------------------------- */
enum qdq_x_op { QDQ_X_PLAIN = 0, QDQ_X_RMSNORM = 1, QDQ_X_SWIGLU = 2, QDQ_X_MUL = 3 };
enum qdq_y_op { QDQ_Y_STORE = 0, QDQ_Y_ADD = 1, QDQ_Y_SILU = 2 };
typedef struct qdq_gemv_opts {
    int32_t x_op;
    int32_t y_op;
    const float *x2;
    const float *norm_w;
    float eps;
    int32_t reserved;
    int64_t *argmax;
} qdq_gemv_opts;
int qdq_plan_create_ex(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n,
                       int batch, qdq_plan **plan_out);
int qdq_plan_run(qdq_plan *plan, qdq_stream_t stream);
/* The same run with host I/O: copies x_host (every distinct x buffer of the
 * plan, concatenated in order of first use, each [batch][cols]) to the plan's x
 * buffers, runs, and copies every GEMV's y (concatenated in descriptor order)
 * into y_host. Host buffers should be pinned. Byte counts are returned through
 * h2d_bytes / d2h_bytes when non-NULL. */
int qdq_plan_run_io(qdq_plan *plan, const float *x_host, float *y_host, qdq_stream_t stream,
                    int64_t *h2d_bytes, int64_t *d2h_bytes);
int qdq_plan_reset(qdq_plan *plan, qdq_stream_t stream);
void qdq_plan_destroy(qdq_plan *plan);
/* Number of kernel launches one qdq_plan_run makes (1). */
int qdq_plan_launches(const qdq_plan *plan);

/* ---------------------------------------------------------------------------
 * qdq_gemv_levels_noalloc: the same computation as a plan built from (descs,
 * level, n, batch) and run once, for callers that cannot allocate device
 * memory (a host framework that owns the whole memory budget, a serving loop
 * that must not call the allocator, a process whose allocations all go through
 * another component). It calls no cudaMalloc or other allocating routine: the
 * level counters live in a 512-byte array in the library's module memory,
 * which every GPU that loads the library keeps until exit. No counterpart on
 * the pages: this is a deployment variant of the plan launch.
 * Limits: at most 128 levels (QDQ_ERR_LIMIT), 192 GEMVs, batch <= 8.
 * The array is shared by every call; each call clears the counters it uses on
 * `stream` first. Calls whose kernels overlap on the GPU race on the array, so
 * serialise them (one stream, or events). The first call on a device looks up
 * the array's device address with that device current; make that first call
 * before any stream capture.
 * ------------------------------------------------------------------------- */
int qdq_gemv_levels_noalloc(const qdq_gemv_desc *descs, const int *level, int n, int batch,
                            qdq_stream_t stream);

/* ---------------------------------------------------------------------------
 * qdq_rope_attention: the attention block of one decode position
 * ("S21 The Capstone: picoLM, in Python", section 4, model_forward, and section
 * 3 for the RoPE layout; "PETIT", How the pieces match: RoPE base, per head).
 *   1. RoPE in the interleaved layout: within each head, the pair
 *      (v[2i], v[2i+1]) of q and of k turns by pos * rope_base^(-2i/head_dim).
 *   2. The cache is fp16: the turned k and the v of this position are rounded
 *      to fp16 (to nearest even) and stored at row pos of k_cache / v_cache.
 *   3. For each query head h, with KV head g = h / (n_heads / n_kv_heads):
 *      out_h = sum_{t <= pos} p_t v_t, p = softmax_t(k_t . q_h / sqrt(head_dim)),
 *      every k_t, v_t in its fp16 value. Online softmax in fp32 (no score array).
 * q: [n_heads * head_dim]; k, v: [n_kv_heads * head_dim]; out: [n_heads *
 * head_dim], fp32 device buffers. k_cache, v_cache: [max_seq][n_kv_heads *
 * head_dim] fp16 bit patterns, device, owned by the caller; rows < pos must hold
 * earlier positions. head_dim even and <= 256, n_heads a multiple of n_kv_heads,
 * 0 <= pos < max_seq (else QDQ_ERR_SHAPE). One launch of n_heads CTAs.
 * ------------------------------------------------------------------------- */
int qdq_rope_attention(const float *q, const float *k, const float *v, uint16_t *k_cache,
                       uint16_t *v_cache, float *out, int n_heads, int n_kv_heads, int head_dim,
                       int pos, int max_seq, float rope_base, qdq_stream_t stream);

/* ---------------------------------------------------------------------------
 * A one-token forward pass of a Llama-architecture model over block-quantised
 * weights ("S21 The Capstone: picoLM, in Python", section 4, model_forward(m,
 * token, pos)): h = the token's embedding row (decoded); per layer
 *   h += Wo attention(rope(Wq n), rope(Wk n), Wv n),  n = rmsnorm(h, attn_norm)
 *   h += Wdown (silu(Wgate n') * Wup n'),              n' = rmsnorm(h, ffn_norm)
 * then logits = Wout rmsnorm(h, output_norm) and their argmax.
 * The embedding's row length in bytes must be a multiple of 16 (QDQ_ERR_ALIGN).
 * Weights are out x in (rows x cols) blocks of any of the four types, device
 * memory owned by the caller, which must outlive the model. layer.w[] and
 * layer.type[] are in the order q, k, v, o, gate, up, down with shapes q, o:
 * dim x dim; k, v: kv x dim (kv = n_kv_heads * dim / n_heads); gate, up:
 * hidden x dim; down: dim x hidden. Norm weights are fp32 device vectors [dim].
 * The model allocates its activations, the fp16 key/value cache
 * ([n_layers][max_seq][kv] each) and one plan in create, and frees them in
 * destroy. A forward call runs 2 launches on `stream`: the embedding row's
 * decode, then one plan of every layer's levels (q/k/v with the attention norm;
 * attention; o with the residual; gate/up with the FFN norm, the gate stored
 * through silu when dim <= 4096; down reading gate * up, or silu(gate) * up
 * when wider, with the residual) and the head with its argmax. Positions must
 * be run in order 0, 1, ... (a position reads the cache rows before it).
 * qdq_llama_buffers returns the device addresses of the logits [vocab], argmax
 * (one int64), the residual stream h [dim] and the two caches.
 * ------------------------------------------------------------------------- */
typedef struct qdq_llama_config {
    int32_t dim, hidden, n_layers, n_heads, n_kv_heads, vocab, max_seq, reserved;
    float rope_base; /* 10000 in PETIT */
    float norm_eps;  /* rmsnorm epsilon */
} qdq_llama_config;
typedef struct qdq_llama_layer {
    const void *w[7];
    int32_t type[7];
    int32_t reserved;
    const float *attn_norm;
    const float *ffn_norm;
} qdq_llama_layer;
typedef struct qdq_llama qdq_llama;
int qdq_llama_create(const qdq_llama_config *cfg, const void *token_embd, int embd_type,
                     const qdq_llama_layer *layers, const float *output_norm, const void *output,
                     int output_type, qdq_llama **model_out);
int qdq_llama_forward(qdq_llama *model, int token, int pos, qdq_stream_t stream);
int qdq_llama_buffers(const qdq_llama *model, float **logits, int64_t **argmax, float **hidden,
                      uint16_t **k_cache, uint16_t **v_cache);
int qdq_llama_launches(const qdq_llama *model);
void qdq_llama_destroy(qdq_llama *model);

/* ---------------------------------------------------------------------------
 * qdq_quantize: fp32 values -> PETIT q8_0 or q4_0 blocks, the exporter's step
 * ("PETIT", What makes it fast & small; How the pieces match: q8_0 = fp32 scale
 * + 32 int8, q4_0 = fp16 scale + 16 nibble bytes read as (q - 8) * d, low
 * nibbles = weights 0..15, values zero-padded to a multiple of 32).
 * The scale rule is not on the pages; this library's reading, per block of 32:
 *   q8_0: d = amax / 127, q = clamp(rint(x / d), -127, 127)   (q = 0 if d = 0)
 *   q4_0: d = fp16(amax / 7), q = clamp(rint(x / d) + 8, 0, 15) (q = 8 if d = 0)
 * with amax = max |x| over the block and every operation in binary32 (the
 * division correctly rounded, rint halving to even), so the codes are those of
 * any CPU that follows the same steps. A q4_0 block whose amax / 7 exceeds the
 * fp16 range (amax > 458528) gets d = inf, which the format cannot represent:
 * its weights decode to NaN. x: n fp32 (device); blocks: ceil(n/32)
 * blocks (device). Both 16-byte aligned. Asynchronous on `stream`.
 * ------------------------------------------------------------------------- */
int qdq_quantize(int type, const float *x, int64_t n, void *blocks, qdq_stream_t stream);

/* ---------------------------------------------------------------------------
 * GGUF container, read from memory (for instance a mapped file): header,
 * metadata, tensor index ("S21 The Capstone: picoLM, in Python", section 1:
 * a header, self-describing metadata, a tensor index of (name, shape, type,
 * offset), padding to general.alignment, then one blob; each tensor is a byte
 * range at a known offset). Host-only, no device work; every read is bounds
 * checked (QDQ_ERR_FORMAT for a bad magic or version, a truncated file, an
 * offset that is not a multiple of the alignment or runs past the end).
 * qdq_gguf_parse fills up to max_tensors entries (QDQ_ERR_LIMIT if the file has
 * more) with the tensors' names, dims (dims[0] innermost: the row length),
 * GGUF type code, the library type that decodes it (QDQ_Q4_0 for type 2,
 * QDQ_Q5_0 for 6, QDQ_Q5_1 for 7, QDQ_Q8_0_GGML for 8, QDQ_Q2_K for 10,
 * QDQ_Q3_K for 11, QDQ_Q4_K for 12, QDQ_Q5_K for 13, QDQ_Q6_K for 14, else 0),
 * absolute byte offset and size.
 * qdq_gguf_find_kv locates a metadata value: its GGUF value type and the byte
 * offset of the value (QDQ_ERR_NOT_FOUND if the key is absent).
 * ------------------------------------------------------------------------- */
typedef struct qdq_gguf_tensor {
    char name[96];
    int32_t n_dims;
    int32_t ggml_type;
    int32_t qdq_type;
    int32_t reserved;
    int64_t dims[4];
    int64_t offset;
    int64_t bytes;
} qdq_gguf_tensor;
int qdq_gguf_parse(const void *file, int64_t size, qdq_gguf_tensor *tensors, int max_tensors,
                   int *n_tensors, int64_t *data_offset, uint32_t *alignment);
int qdq_gguf_find_kv(const void *file, int64_t size, const char *key, uint32_t *value_type,
                     int64_t *value_offset);

/* ---------------------------------------------------------------------------
 * Device status: synchronises `stream`, returns the first device-side error
 * recorded since the last call (QDQ_OK if none) and clears it.
 * ------------------------------------------------------------------------- */
int qdq_get_device_status(qdq_stream_t stream);

/* Runs the library's bounded inter-CTA wait on a device flag that nothing sets,
 * with a limit of `timeout_ns` nanoseconds, so that a test can see a wait run
 * out without a hang: afterwards qdq_get_device_status() returns
 * QDQ_ERR_TIMEOUT. */
int qdq_selftest_wait_timeout(int64_t timeout_ns, qdq_stream_t stream);

/* Number of streaming multiprocessors the library sizes its grids by. */
int qdq_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* QDQ_H */
