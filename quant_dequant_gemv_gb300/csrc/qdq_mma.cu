// qdq_mma.cu -- batched dequant-GEMV on the tensor cores (tcgen05), batch >= 9.
#include "qdq_internal.h"

namespace qdq {

int launch_mma_gemv(int, const void *, int64_t, int64_t, const float *, float *, int, cudaStream_t, int) {
    return QDQ_ERR_LIMIT;
}

int take_status_mma() { return QDQ_OK; }

}  // namespace qdq
