// qdq_internal.h -- host-side declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "qdq.h"

namespace qdq {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    bool ok = false;
};

// Cached per device; ok == false when the current device is not sm_103.
const DeviceInfo &current_device(int *status);

// Argument checks shared by every entry point that takes GEMV descriptors
// (qdq_api.cu): shapes and device pointers, and the plan level sequence.
int check_descs(const qdq_gemv_desc *descs, int n, int batch, int device);
int check_levels(const int *level, int n, int max_levels, int *nlevels);

int launch_dequant(int type, const void *blocks, int64_t n, float *out, cudaStream_t stream, int sm_count);
int launch_quantize(int type, const float *x, int64_t n, void *blocks, cudaStream_t stream, int sm_count);
// The further GGUF formats (Q5_0, Q5_1, ggml q8_0, Q2_K): qdq_gemv_more.cu.
bool is_more_type(int type);
int launch_gemv_more(int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y, int batch,
                     cudaStream_t stream, int sm_count);

// The streaming (CUDA-core) GEMV over a list of GEMVs grouped in dependency levels.
struct StreamPlanHost;  // opaque: the packed kernel arguments
// opts (may be NULL: every GEMV plain) and amax_slot (two zeroed 64-bit words,
// needed when an option asks for an argmax) as for qdq_plan_create_ex.
int stream_plan_build(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n,
                      int batch, unsigned *counters, unsigned long long *amax_slot, int sm_count,
                      StreamPlanHost **out);
int stream_plan_launch(const StreamPlanHost *p, cudaStream_t stream);
// The position attention levels of the plan run at (the next launches).
void stream_plan_set_pos(StreamPlanHost *p, int pos);

// A plan level that is not a GEMV: the attention block of one position, one query
// head per CTA (qdq_stream1.cu, attend). Packed as a descriptor of type
// kTypeAttn (64) with W = the key cache, x = q, y = the output, rows = query
// heads, cols = head_dim, and its options holding x2 = k, norm_w = v, argmax =
// the value cache, reserved = KV heads, eps = the RoPE base. Alone in its level.
constexpr int kPlanAttnType = 64;
// qdq_plan_create_ex for plans that also hold attention levels: the GEMVs are
// checked as there; the attention descriptors are the caller's (the model's).
int plan_create_with_attention(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n,
                               qdq_plan **plan_out);
int plan_set_pos(qdq_plan *plan, int pos);
void stream_plan_free(StreamPlanHost *p);
int stream_plan_nlevels(const StreamPlanHost *p);
int stream_launch_levels_inplace(const qdq_gemv_desc *descs, const int *level, int n, int batch,
                                 unsigned *counters, int sm_count, cudaStream_t stream);

int take_status_stream();
// The streaming kernel (qdq_stream1.cu) at batch width bt (1, 2, 4 or 8): runs the
// argument block packed by the plan functions above.
int stream1_launch(const void *args, bool big, bool cooperative, int grid, int bt, bool attn, cudaStream_t stream);
int take_status_stream1();
int launch_wait_selftest(int64_t limit_ns, cudaStream_t stream);

// The tensor-core batched GEMV (single GEMVs from mma_min_batch on; it accepts any
// batch >= kMmaMinBatch).
int launch_mma_gemv(int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y,
                    int batch, cudaStream_t stream, int sm_count);
int take_status_mma();

// While a caller's stream is being captured into a CUDA graph, one-time setup calls
// (kernel attributes, occupancy queries, memory-pool creation) would invalidate a
// capture in global mode; this scope relaxes the calling thread's capture mode for
// them. Stream operations issued inside it are still captured.
struct RelaxedCaptureScope {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    RelaxedCaptureScope() { cudaThreadExchangeStreamCaptureMode(&mode); }
    ~RelaxedCaptureScope() { cudaThreadExchangeStreamCaptureMode(&mode); }
    RelaxedCaptureScope(const RelaxedCaptureScope &) = delete;
    RelaxedCaptureScope &operator=(const RelaxedCaptureScope &) = delete;
};

constexpr int kMaxPlanDescs = 192;
constexpr int kMaxPlanLevels = 128;
constexpr int kMaxGroupDescs = 8;
constexpr int kStreamMaxBatch = 8;  // streaming kernel (plans, groups, small single GEMVs)
constexpr int kMmaMinBatch = 4;     // the tensor-core path takes batches from this one on
// Single GEMVs run on the tensor cores from this batch on (measured crossover with
// the CUDA-core streaming kernel on GB300: Q4_K and Q6_K stream faster up to batch
// 4, which the streaming kernel's four-column instantiation covers; from batch 5 it
// runs its eight-column instantiation and the tensor cores win. For the 32-weight
// block formats q8_0 and q4_0 the tensor cores are faster already at batch 4).
inline int mma_min_batch(int type) { return (type == QDQ_Q8_0 || type == QDQ_Q4_0) ? 4 : 5; }

}  // namespace qdq
