// qdq_noalloc.cu -- the dependency-level GEMV launch for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a fixed memory
// budget handed to it by a host framework, code that must not touch the
// allocator once a serving loop is running, or code linked into a process whose
// allocations all go through another component. qdq_plan_create allocates the
// plan's level counters with cudaMalloc; qdq_gemv_levels_noalloc runs the same
// persistent kernel with its counters in a file-scope device array instead.
//
// The array holds kNoAllocMaxLevels counters (512 bytes). Every GPU that loads
// the library keeps it until the process exits, and every call shares it: the
// call clears the counters it uses on `stream` before the launch, and two calls
// whose kernels overlap on the GPU race on the array.
#include <mutex>

#include "qdq_internal.h"

namespace qdq {

constexpr int kNoAllocMaxLevels = 128;

static __device__ __align__(256) unsigned s_noalloc_level_counters[kNoAllocMaxLevels];

// Device address of the array, looked up once per device with that device current.
static unsigned *s_counters_addr[64];
static std::mutex s_counters_mu;

static int counters_for_device(int device, unsigned **out) {
    std::lock_guard<std::mutex> lock(s_counters_mu);
    if (s_counters_addr[device] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, s_noalloc_level_counters) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return QDQ_ERR_CUDA;
        }
        s_counters_addr[device] = (unsigned *)p;
    }
    *out = s_counters_addr[device];
    return QDQ_OK;
}

}  // namespace qdq

using namespace qdq;

extern "C" int qdq_gemv_levels_noalloc(const qdq_gemv_desc *descs, const int *level, int n, int batch,
                                       qdq_stream_t stream) {
    if (descs == nullptr || level == nullptr) return QDQ_ERR_PTR;
    if (n < 1 || n > kMaxPlanDescs) return QDQ_ERR_LIMIT;
    if (batch < 1) return QDQ_ERR_SHAPE;
    if (batch > kStreamMaxBatch) return QDQ_ERR_LIMIT;
    int nlevels = 0;
    int rc = check_levels(level, n, kNoAllocMaxLevels, &nlevels);
    if (rc) return rc;
    const DeviceInfo &dev = current_device(&rc);
    if (rc) return rc;
    if ((rc = check_descs(descs, n, batch, dev.device))) return rc;
    unsigned *counters = nullptr;
    if ((rc = counters_for_device(dev.device, &counters))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(counters, 0, sizeof(unsigned) * nlevels, s) != cudaSuccess) {
        cudaGetLastError();
        return QDQ_ERR_CUDA;
    }
    return stream_launch_levels_inplace(descs, level, n, batch, counters, dev.sm_count, s);
}
