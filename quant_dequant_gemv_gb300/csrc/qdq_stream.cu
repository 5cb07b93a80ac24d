// qdq_stream.cu -- host side of the CUDA-core streaming path: packing GEMV
// descriptors and dependency levels into the persistent kernel's argument block
// (qdq_stream1.cu holds the kernel), the plan objects built on it, and the
// bounded-wait self-test.
//
// "S21 The Capstone: picoLM, in Python", section 4 (model_forward: the per-layer
// projections of a decode step, each reading the previous one's output, which
// is what the dependency levels encode); "PETIT" (gemv_q8 / gemv_q4, weights
// stored out x in).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "qdq_stream_common.cuh"

namespace qdq {

static __device__ int s_status_stream;

// Counter wait with nothing to release it: the wait gives up after limit_ns and
// records QDQ_ERR_TIMEOUT in the status word.
__global__ void wait_selftest_kernel(const unsigned *flag, int64_t limit_ns) {
    wait_counter(flag, 1u, &s_status_stream, (uint64_t)limit_ns);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct StreamPlanHost {
    int bt;
    int grid;
    bool cooperative;
    size_t args_bytes;
    void *args;  // StreamArgs<...>
    bool big;
    bool attn;  // the plan has attention levels
};

#ifdef QDQ_TRACE
static unsigned long long *s_trace = nullptr;
#endif

template <int MAXD, int MAXL>
static void fill_args(StreamArgs<MAXD, MAXL> *A, const qdq_gemv_desc *descs, const qdq_gemv_opts *opts,
                      const int *level, int n, int batch, unsigned *counters, unsigned long long *amax_slot) {
    memset(A, 0, sizeof(*A));
#ifdef QDQ_TRACE
    A->trace = s_trace;
#endif
    A->ndesc = n;
    A->batch = batch;
    A->counters = counters;
    int L = 0;
    A->level_start[0] = 0;
    for (int i = 0; i < n; ++i) {
        const int lv = level ? level[i] : 0;
        while (L < lv) A->level_start[++L] = i;
    }
    A->nlevels = L + 1;
    A->level_start[L + 1] = n;
    for (int i = 0; i < n; ++i) {
        DevDesc &d = A->d[i];
        DescEx &e = A->ex[i];
        if (descs[i].type == kTypeAttn) {  // packed as kPlanAttnType describes
            d.type = kTypeAttn;
            d.x = descs[i].x;
            d.y = descs[i].y;
            d.rows = descs[i].rows;
            d.cols = (int32_t)descs[i].cols;
            d.nkv = opts[i].reserved;
            e.kc = (uint16_t *)descs[i].W;
            e.vc = (uint16_t *)opts[i].argmax;
            e.x2 = opts[i].x2;
            e.nw = opts[i].norm_w;
            for (int p = 0; p < d.cols / 2 && p < kMaxRopePairs; ++p)
                A->rope_f[p] = std::pow((double)opts[i].eps, -2.0 * p / (double)d.cols);
            continue;
        }
        d.W = (const uint8_t *)descs[i].W;
        d.x = descs[i].x;
        d.y = descs[i].y;
        d.rows = descs[i].rows;
        d.cols = (int32_t)descs[i].cols;
        d.type = descs[i].type;
        d.rb = (int32_t)((descs[i].cols / blk_weights(d.type)) * blk_bytes(d.type));
        if (opts) {
            d.ops = (opts[i].x_op & 15) | ((opts[i].y_op & 15) << 4) | (opts[i].argmax ? 256 : 0);
            e.x2 = opts[i].x2;
            e.nw = opts[i].norm_w;
            e.eps = opts[i].eps;
            if (opts[i].argmax) {
                A->amax_slot = amax_slot;
                A->amax_y = descs[i].y;
                A->amax_out = (long long *)opts[i].argmax;
            }
        }
    }
    // staged copy kinds per (level, x)
    for (int lv = 0; lv < A->nlevels; ++lv) {
        for (int i = A->level_start[lv]; i < A->level_start[lv + 1]; ++i) {
            int kinds = 0;
            for (int k = A->level_start[lv]; k < A->level_start[lv + 1]; ++k)
                if (A->d[k].x == A->d[i].x && A->d[k].type != kTypeAttn) kinds |= 1 << x_kind(A->d[k].type);
            A->d[i].kinds = kinds;
        }
    }
}

static int bt_of(int batch) { return batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }

int stream_plan_build(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n, int batch,
                      unsigned *counters, unsigned long long *amax_slot, int sm_count, StreamPlanHost **out) {
    StreamPlanHost *p = new (std::nothrow) StreamPlanHost();
    if (!p) return QDQ_ERR_CUDA;
    p->bt = bt_of(batch);
    p->grid = sm_count;
    const int nlev = level ? level[n - 1] + 1 : 1;
    p->attn = false;
    // the model's instantiation (plan-sized arguments): attention levels, silu
    // applied at the store, or x * x2 staged
    for (int i = 0; i < n; ++i)
        p->attn = p->attn || descs[i].type == kTypeAttn ||
                  (opts != nullptr && (opts[i].y_op == QDQ_Y_SILU || opts[i].x_op == QDQ_X_MUL));
    p->big = n > kMaxGroupDescs || nlev > 1 || p->attn;
    p->cooperative = nlev > 1;
    if (p->big) {
        using A = StreamArgs<kMaxPlanDescs, kMaxPlanLevels>;
        A *args = (A *)malloc(sizeof(A));
        if (!args) { delete p; return QDQ_ERR_CUDA; }
        fill_args(args, descs, opts, level, n, batch, counters, amax_slot);
        p->args = args;
        p->args_bytes = sizeof(A);
    } else {
        using A = StreamArgs<kMaxGroupDescs, 1>;
        A *args = (A *)malloc(sizeof(A));
        if (!args) { delete p; return QDQ_ERR_CUDA; }
        fill_args(args, descs, opts, level, n, batch, counters, amax_slot);
        p->args = args;
        p->args_bytes = sizeof(A);
    }
    *out = p;
    return QDQ_OK;
}

void stream_plan_set_pos(StreamPlanHost *p, int pos) {
    if (p->big)
        ((StreamArgs<kMaxPlanDescs, kMaxPlanLevels> *)p->args)->attn_pos = pos;
    else
        ((StreamArgs<kMaxGroupDescs, 1> *)p->args)->attn_pos = pos;
}

int stream_plan_launch(const StreamPlanHost *p, cudaStream_t stream) {
    return stream1_launch(p->args, p->big, p->cooperative, p->grid, p->bt, p->attn, stream);
}

// Multi-level launch with caller-provided level counters and no heap use: the
// kernel arguments live on this function's stack (about 10 KiB).
int stream_launch_levels_inplace(const qdq_gemv_desc *descs, const int *level, int n, int batch,
                                 unsigned *counters, int sm_count, cudaStream_t stream) {
    using A = StreamArgs<kMaxPlanDescs, kMaxPlanLevels>;
    A args;
    StreamPlanHost p;
    p.bt = bt_of(batch);
    p.grid = sm_count;
    p.big = true;
    p.cooperative = true;
    p.attn = false;
    p.args = &args;
    p.args_bytes = sizeof(A);
    fill_args(&args, descs, nullptr, level, n, batch, counters, nullptr);
    return stream_plan_launch(&p, stream);
}

void stream_plan_free(StreamPlanHost *p) {
    if (!p) return;
    free(p->args);
    delete p;
}

int stream_plan_nlevels(const StreamPlanHost *p) {
    return p->big ? ((StreamArgs<kMaxPlanDescs, kMaxPlanLevels> *)p->args)->nlevels : 1;
}

#ifdef QDQ_TRACE
}  // namespace qdq
extern "C" void qdq_debug_set_trace(unsigned long long *buf) { qdq::s_trace = buf; }
namespace qdq {
#endif

int take_status_stream() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, s_status_stream, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(s_status_stream, &zero, sizeof(int)) != cudaSuccess) return QDQ_ERR_CUDA;
    return v;
}

int launch_wait_selftest(int64_t limit_ns, cudaStream_t stream) {
    unsigned *flag = nullptr;
    if (cudaMallocAsync((void **)&flag, sizeof(unsigned), stream) != cudaSuccess) return QDQ_ERR_CUDA;
    cudaMemsetAsync(flag, 0, sizeof(unsigned), stream);
    wait_selftest_kernel<<<1, 1, 0, stream>>>(flag, limit_ns);
    const cudaError_t e = cudaGetLastError();
    cudaFreeAsync(flag, stream);
    return e == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
}

}  // namespace qdq
