// qdq_api.cu -- the extern "C" boundary of libqdq (declared in include/qdq.h):
// argument checks, device checks, dispatch to the kernels, plans, status.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "qdq_decode.cuh"
#include "qdq_internal.h"

namespace qdq {

const DeviceInfo &current_device(int *status) {
    static DeviceInfo cache[64];
    static std::mutex mu;
    static DeviceInfo bad;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        *status = QDQ_ERR_CUDA;
        return bad;
    }
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &d = cache[dev];
    if (d.device != dev) {
        int maj = 0, min = 0, sms = 0;
        if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            *status = QDQ_ERR_CUDA;
            return bad;
        }
        d.cc_major = maj;
        d.cc_minor = min;
        d.sm_count = sms;
        d.ok = (maj == 10 && min == 3);
        d.device = dev;
    }
    *status = d.ok ? QDQ_OK : QDQ_ERR_DEVICE;
    return d;
}

// The main four formats (every path) and the further GGUF ones (dequant, qdq_gemv).
static bool main_type(int type) {
    return type == QDQ_Q4_0 || type == QDQ_Q8_0 || type == QDQ_Q4_K || type == QDQ_Q6_K;
}
static int check_type(int type) { return (main_type(type) || is_more_type(type)) ? QDQ_OK : QDQ_ERR_TYPE; }

// Device (or managed) memory of the current device, 16-byte aligned.
static int check_dev_ptr(const void *p, int device) {
    if (p == nullptr) return QDQ_ERR_PTR;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_PTR;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return QDQ_ERR_PTR;
    if (attr.type == cudaMemoryTypeDevice && attr.device != device) return QDQ_ERR_PTR;
    if (((uintptr_t)p & 15) != 0) return QDQ_ERR_ALIGN;
    return QDQ_OK;
}

static int check_gemv_shape(int type, int64_t rows, int64_t cols, int batch) {
    int rc = check_type(type);
    if (rc) return rc;
    if (rows < 0 || cols < 0 || batch < 1) return QDQ_ERR_SHAPE;
    if (cols % qdq_block_weights(type)) return QDQ_ERR_SHAPE;
    if (rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 30)) return QDQ_ERR_SHAPE;
    return QDQ_OK;
}

static int check_gemv_ptrs(const void *W, const float *x, float *y, int device) {
    int rc = check_dev_ptr(W, device);
    if (!rc) rc = check_dev_ptr(x, device);
    if (!rc) rc = check_dev_ptr(y, device);
    return rc;
}

// Descriptors of a group or plan: shapes, pointers, and agreement on shared x.
int check_descs(const qdq_gemv_desc *descs, int n, int batch, int device) {
    if (descs == nullptr || n < 0) return QDQ_ERR_PTR;
    for (int i = 0; i < n; ++i) {
        if (!main_type(descs[i].type)) return QDQ_ERR_TYPE;  // groups and plans: the main four
        int rc = check_gemv_shape(descs[i].type, descs[i].rows, descs[i].cols, batch);
        if (rc) return rc;
        if (descs[i].rows == 0 || descs[i].cols == 0) return QDQ_ERR_SHAPE;
        if ((rc = check_gemv_ptrs(descs[i].W, descs[i].x, descs[i].y, device))) return rc;
    }
    // GEMVs that read the same x must agree on its length
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < i; ++k)
            if (descs[k].x == descs[i].x && descs[k].cols != descs[i].cols) return QDQ_ERR_SHAPE;
    return QDQ_OK;
}


// Level indices of a plan: start at 0 and never skip or go back. *nlevels gets
// the level count; more than max_levels gives QDQ_ERR_LIMIT.
int check_levels(const int *level, int n, int max_levels, int *nlevels) {
    if (level[0] != 0) return QDQ_ERR_SHAPE;
    for (int i = 1; i < n; ++i)
        if (level[i] != level[i - 1] && level[i] != level[i - 1] + 1) return QDQ_ERR_SHAPE;
    *nlevels = level[n - 1] + 1;
    return *nlevels > max_levels ? QDQ_ERR_LIMIT : QDQ_OK;
}

}  // namespace qdq

using namespace qdq;

struct qdq_plan {
    StreamPlanHost *host = nullptr;
    unsigned *counters = nullptr;
    unsigned long long *amax = nullptr;  // argmax slot (plans with an argmax option)
    int device = -1;
    int n = 0, batch = 1, nlevels = 1;
    std::vector<qdq_gemv_desc> descs;
};

extern "C" {

int qdq_block_bytes(int type) { return check_type(type) ? -1 : fmt_bytes(type); }

int qdq_block_weights(int type) { return check_type(type) ? -1 : fmt_weights(type); }

const char *qdq_status_string(int status) {
    switch (status) {
        case QDQ_OK: return "ok";
        case QDQ_ERR_TYPE: return "unknown block type";
        case QDQ_ERR_SHAPE: return "invalid shape (negative size, cols/n not a multiple of the block, or batch < 1)";
        case QDQ_ERR_ALIGN: return "pointer not 16-byte aligned";
        case QDQ_ERR_PTR: return "NULL or non-device pointer";
        case QDQ_ERR_CUDA: return "CUDA runtime or launch failure";
        case QDQ_ERR_TIMEOUT: return "a device-side bounded wait ran out";
        case QDQ_ERR_DEVICE: return "current device is not sm_103 (GB300)";
        case QDQ_ERR_LIMIT: return "too many GEMVs or levels for a plan, or batch too large for it";
        case QDQ_ERR_FORMAT: return "malformed or truncated GGUF data";
        case QDQ_ERR_NOT_FOUND: return "no such GGUF metadata key";
        case QDQ_ERR_BOUNDS: return "device-side index or alignment check failed (debug build)";
        default: return "unknown status";
    }
}

int qdq_device_sm_count(void) {
    int st;
    const DeviceInfo &d = current_device(&st);
    return st == QDQ_OK ? d.sm_count : st;
}

int qdq_dequant_async(int type, const void *blocks, int64_t n, float *out_f32, qdq_stream_t stream) {
    int rc = check_type(type);
    if (rc) return rc;
    if (n < 0 || n % qdq_block_weights(type)) return QDQ_ERR_SHAPE;
    if (n == 0) return QDQ_OK;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    if ((rc = check_dev_ptr(blocks, dev.device)) || (rc = check_dev_ptr(out_f32, dev.device))) return rc;
    return launch_dequant(type, blocks, n, out_f32, (cudaStream_t)stream, dev.sm_count);
}

int qdq_dequant(int type, const void *blocks, int64_t n, float *out_f32) {
    return qdq_dequant_async(type, blocks, n, out_f32, nullptr);
}

static int run_stream_once(const qdq_gemv_desc *descs, int n, int batch, cudaStream_t stream, int sm_count) {
    StreamPlanHost *p = nullptr;
    int rc = stream_plan_build(descs, nullptr, nullptr, n, batch, nullptr, nullptr, sm_count, &p);
    if (rc) return rc;
    rc = stream_plan_launch(p, stream);
    stream_plan_free(p);
    return rc;
}

int qdq_gemv(int type, const void *W, int64_t rows, int64_t cols, const float *x, float *y, int batch,
             qdq_stream_t stream) {
    int rc = check_gemv_shape(type, rows, cols, batch);
    if (rc) return rc;
    if (rows == 0) return QDQ_OK;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    if ((rc = check_gemv_ptrs(W, x, y, dev.device))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (cols == 0)
        return cudaMemsetAsync(y, 0, (size_t)batch * rows * sizeof(float), s) == cudaSuccess ? QDQ_OK : QDQ_ERR_CUDA;
    if (is_more_type(type)) return launch_gemv_more(type, W, rows, cols, x, y, batch, s, dev.sm_count);
    if (batch >= mma_min_batch(type)) {
        rc = launch_mma_gemv(type, W, rows, cols, x, y, batch, s, dev.sm_count);
        if (rc != QDQ_ERR_LIMIT) return rc;
        // shapes the tensor-core path does not take: batch slices of <= 8
        for (int b0 = 0; b0 < batch; b0 += kStreamMaxBatch) {
            const int nb = batch - b0 < kStreamMaxBatch ? batch - b0 : kStreamMaxBatch;
            qdq_gemv_desc d = {type, 0, W, rows, cols, x + (int64_t)b0 * cols, y + (int64_t)b0 * rows};
            if ((rc = run_stream_once(&d, 1, nb, s, dev.sm_count))) return rc;
        }
        return QDQ_OK;
    }
    qdq_gemv_desc d = {type, 0, W, rows, cols, x, y};
    return run_stream_once(&d, 1, batch, s, dev.sm_count);
}

int qdq_gemv_group(const qdq_gemv_desc *descs, int n, int batch, qdq_stream_t stream) {
    if (n == 0) return QDQ_OK;
    if (n < 0 || n > kMaxGroupDescs) return QDQ_ERR_LIMIT;
    if (batch < 1) return QDQ_ERR_SHAPE;
    if (batch > kStreamMaxBatch) return QDQ_ERR_LIMIT;
    int rc;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    if ((rc = check_descs(descs, n, batch, dev.device))) return rc;
    return run_stream_once(descs, n, batch, (cudaStream_t)stream, dev.sm_count);
}

int qdq_plan_create(const qdq_gemv_desc *descs, const int *level, int n, int batch, qdq_plan **plan_out) {
    return qdq_plan_create_ex(descs, nullptr, level, n, batch, plan_out);
}

// The rules of qdq_gemv_opts (include/qdq.h).
static int check_opts(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n, int batch,
                      int device, bool *has_argmax) {
    *has_argmax = false;
    if (opts == nullptr) return QDQ_OK;
    int rc = QDQ_OK;
    for (int i = 0; i < n && !rc; ++i) {
        const qdq_gemv_opts &o = opts[i];
        if (o.x_op < QDQ_X_PLAIN || o.x_op > QDQ_X_MUL || o.y_op < QDQ_Y_STORE || o.y_op > QDQ_Y_SILU)
            return QDQ_ERR_SHAPE;
        // silu at the store needs each row's whole sum in one flush: batch 1 and
        // whole-row tiles in one x window (two 2048-column chunks at least); both
        // options run in the batch-1 kernel that also holds attention levels
        if (o.y_op == QDQ_Y_SILU && (batch != 1 || descs[i].cols > 4096)) return QDQ_ERR_SHAPE;
        if (o.x_op == QDQ_X_MUL && batch != 1) return QDQ_ERR_SHAPE;
        if (o.x_op == QDQ_X_RMSNORM) {
            if (!(o.eps >= 0.0f) || o.eps > 1.0f) return QDQ_ERR_SHAPE;
            rc = check_dev_ptr(o.norm_w, device);
        }
        if (!rc && (o.x_op == QDQ_X_SWIGLU || o.x_op == QDQ_X_MUL)) rc = check_dev_ptr(o.x2, device);
        if (!rc && o.argmax) {
            if (*has_argmax || batch != 1 || level[i] != level[n - 1] || descs[i].cols > 8192) return QDQ_ERR_SHAPE;
            if (descs[i].rows > 0xFFFFFFFFll) return QDQ_ERR_SHAPE;
            rc = check_dev_ptr(o.argmax, device);
            *has_argmax = true;
        }
        // GEMVs of one level reading the same x stage it once: same x option
        for (int k = 0; k < i && !rc; ++k)
            if (level[k] == level[i] && descs[k].x == descs[i].x &&
                (opts[k].x_op != o.x_op || ((o.x_op == QDQ_X_SWIGLU || o.x_op == QDQ_X_MUL) && opts[k].x2 != o.x2) ||
                 (o.x_op == QDQ_X_RMSNORM && (opts[k].norm_w != o.norm_w || opts[k].eps != o.eps))))
                return QDQ_ERR_SHAPE;
    }
    return rc;
}

// Plan creation; with allow_attn, descriptors of type kPlanAttnType are attention
// levels packed by the model (qdq_llama.cu) and skip the GEMV checks.
static int plan_create(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n, int batch,
                       bool allow_attn, qdq_plan **plan_out) {
    if (plan_out == nullptr || level == nullptr) return QDQ_ERR_PTR;
    *plan_out = nullptr;
    if (n < 1 || n > kMaxPlanDescs) return QDQ_ERR_LIMIT;
    if (batch < 1) return QDQ_ERR_SHAPE;
    if (batch > kStreamMaxBatch) return QDQ_ERR_LIMIT;
    int nlevels = 0;
    int rc = check_levels(level, n, kMaxPlanLevels, &nlevels);
    if (rc) return rc;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    // the GEMVs (every descriptor unless attention levels are allowed)
    std::vector<qdq_gemv_desc> gd;
    std::vector<qdq_gemv_opts> go;
    std::vector<int> gl;
    for (int i = 0; i < n; ++i) {
        if (allow_attn && descs[i].type == kPlanAttnType) {
            if (batch != 1) return QDQ_ERR_SHAPE;
            continue;
        }
        gd.push_back(descs[i]);
        if (opts) go.push_back(opts[i]);
        gl.push_back(level[i]);
    }
    if ((rc = check_descs(gd.data(), (int)gd.size(), batch, dev.device))) return rc;
    bool has_argmax = false;
    if (!gd.empty() &&
        (rc = check_opts(gd.data(), opts ? go.data() : nullptr, gl.data(), (int)gd.size(), batch, dev.device,
                         &has_argmax)))
        return rc;
    qdq_plan *p = new (std::nothrow) qdq_plan();
    if (!p) return QDQ_ERR_CUDA;
    p->device = dev.device;
    p->n = n;
    p->batch = batch;
    p->nlevels = nlevels;
    p->descs.assign(descs, descs + n);
    auto fail = [&](int code) {
        cudaGetLastError();
        if (p->counters) cudaFree(p->counters);
        if (p->amax) cudaFree(p->amax);
        delete p;
        return code;
    };
    if (cudaMalloc((void **)&p->counters, sizeof(unsigned) * nlevels) != cudaSuccess ||
        cudaMemset(p->counters, 0, sizeof(unsigned) * nlevels) != cudaSuccess)
        return fail(QDQ_ERR_CUDA);
    if (has_argmax && (cudaMalloc((void **)&p->amax, 2 * sizeof(unsigned long long)) != cudaSuccess ||
                       cudaMemset(p->amax, 0, 2 * sizeof(unsigned long long)) != cudaSuccess))
        return fail(QDQ_ERR_CUDA);
    if ((rc = stream_plan_build(descs, opts, level, n, batch, p->counters, p->amax, dev.sm_count, &p->host)))
        return fail(rc);
    *plan_out = p;
    return QDQ_OK;
}

int qdq_plan_create_ex(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n, int batch,
                       qdq_plan **plan_out) {
    return plan_create(descs, opts, level, n, batch, false, plan_out);
}

int qdq_plan_run(qdq_plan *plan, qdq_stream_t stream) {
    if (plan == nullptr) return QDQ_ERR_PTR;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) return QDQ_ERR_DEVICE;
    return stream_plan_launch(plan->host, (cudaStream_t)stream);
}

// Issue copies for a list of (device ptr, bytes) ranges, merging ranges that
// are adjacent both on the device and in the host buffer.
static int copy_ranges(const std::vector<std::pair<char *, size_t>> &ranges, char *host, bool to_device,
                       cudaStream_t s, int64_t *bytes_out) {
    size_t hoff = 0;
    int64_t total = 0;
    size_t i = 0;
    while (i < ranges.size()) {
        char *dptr = ranges[i].first;
        size_t len = ranges[i].second;
        size_t j = i + 1;
        while (j < ranges.size() && ranges[j].first == dptr + len) len += ranges[j++].second;
        const cudaError_t e = to_device ? cudaMemcpyAsync(dptr, host + hoff, len, cudaMemcpyHostToDevice, s)
                                        : cudaMemcpyAsync(host + hoff, dptr, len, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return QDQ_ERR_CUDA;
        }
        hoff += len;
        total += (int64_t)len;
        i = j;
    }
    if (bytes_out) *bytes_out = total;
    return QDQ_OK;
}

int qdq_plan_run_io(qdq_plan *plan, const float *x_host, float *y_host, qdq_stream_t stream, int64_t *h2d_bytes,
                    int64_t *d2h_bytes) {
    if (plan == nullptr || x_host == nullptr || y_host == nullptr) return QDQ_ERR_PTR;
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<std::pair<char *, size_t>> xr, yr;
    for (int i = 0; i < plan->n; ++i) {
        const qdq_gemv_desc &d = plan->descs[i];
        bool seen = false;
        for (int k = 0; k < i && !seen; ++k) seen = plan->descs[k].x == d.x;
        if (!seen) xr.push_back({(char *)d.x, (size_t)plan->batch * d.cols * sizeof(float)});
        yr.push_back({(char *)d.y, (size_t)plan->batch * d.rows * sizeof(float)});
    }
    int rc = copy_ranges(xr, (char *)x_host, true, s, h2d_bytes);
    if (rc) return rc;
    if ((rc = qdq_plan_run(plan, stream))) return rc;
    return copy_ranges(yr, (char *)y_host, false, s, d2h_bytes);
}

int qdq_plan_reset(qdq_plan *plan, qdq_stream_t stream) {
    if (plan == nullptr) return QDQ_ERR_PTR;
    if (cudaMemsetAsync(plan->counters, 0, sizeof(unsigned) * plan->nlevels, (cudaStream_t)stream) != cudaSuccess ||
        (plan->amax && cudaMemsetAsync(plan->amax, 0, 2 * sizeof(unsigned long long), (cudaStream_t)stream) != cudaSuccess)) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return QDQ_OK;
}

void qdq_plan_destroy(qdq_plan *plan) {
    if (plan == nullptr) return;
    stream_plan_free(plan->host);
    if (plan->counters) cudaFree(plan->counters);
    if (plan->amax) cudaFree(plan->amax);
    delete plan;
}

int qdq_plan_launches(const qdq_plan *plan) { return plan ? 1 : 0; }

int qdq_get_device_status(qdq_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    const int a = take_status_stream();
    const int a1 = take_status_stream1();
    const int b = take_status_mma();
    return a != QDQ_OK ? a : a1 != QDQ_OK ? a1 : b;
}

int qdq_selftest_wait_timeout(int64_t timeout_ns, qdq_stream_t stream) {
    if (timeout_ns < 0) return QDQ_ERR_SHAPE;
    int rc;
    current_device(&rc);
    if (rc) return rc;
    return launch_wait_selftest(timeout_ns, (cudaStream_t)stream);
}

}  // extern "C"

namespace qdq {
int plan_create_with_attention(const qdq_gemv_desc *descs, const qdq_gemv_opts *opts, const int *level, int n,
                               qdq_plan **plan_out) {
    return plan_create(descs, opts, level, n, 1, true, plan_out);
}
int plan_set_pos(qdq_plan *plan, int pos) {
    if (plan == nullptr) return QDQ_ERR_PTR;
    stream_plan_set_pos(plan->host, pos);
    return QDQ_OK;
}
}  // namespace qdq
