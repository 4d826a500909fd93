// Chunked prefill against a paged prefix (placeholder until the tensor-core
// kernel lands): reports every shape as not built.
#include "pkv_internal.h"

namespace pkv {

size_t prefill_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int32_t, int32_t, int32_t,
                               int32_t, pkv_dtype)
{
    return 256;
}

cudaError_t launch_prefill(const void *, const int32_t *, int32_t, const pkv_pool &,
                           const int32_t *, int32_t, const int32_t *, int32_t, int32_t, int32_t,
                           int32_t, float, void *, void *, size_t, int32_t *, cudaStream_t,
                           int *unsupported)
{
    *unsupported = 1;
    return cudaSuccess;
}

}  // namespace pkv
