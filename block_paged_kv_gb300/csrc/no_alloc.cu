// Decode attention for callers that cannot allocate device memory.
//
// paged_decode_attention needs a scratch workspace for its split partials,
// which the caller allocates.  Some callers cannot do that where they call us:
// a plug-in living inside a host framework that keeps every byte of device
// memory in its own allocator and hands none out, or a latency-bound serving
// loop that bans cudaMalloc on its hot path (cudaMalloc may synchronize the
// device and may fail under memory pressure).  For them this file keeps the
// scratch in the library's own device image: a fixed array that exists on
// every GPU that loads the library, from load until the process exits.
#include <algorithm>
#include <mutex>

#include <cuda_runtime.h>

#include "pkv.h"

namespace {

// The shared scratch.  Host code must not use this name as a device address
// (on the host it names a stand-in object): the device address comes from
// cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};

// Device address of g_scratch on the current device, looked up on the first
// call made with that device current and remembered afterwards.
pkv_status scratch_for_current_device(void **addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status paged_decode_attention_no_alloc(
    const void *q, int32_t num_q_heads, const pkv_pool *pool, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch, int32_t max_seq_len,
    int32_t window, float scale, void *out, const pkv_prefix_desc *prefix, int32_t *dev_status,
    pkv_stream_t stream)
{
    if (pool == nullptr) return PKV_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const pkv_status st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;
    // the same plan the workspace entry point makes for these sizes
    int64_t len = max_seq_len;
    if (max_blocks_per_seq > 0 && pool->block_size > 0)
        len = std::min<int64_t>(len, static_cast<int64_t>(max_blocks_per_seq) * pool->block_size);
    const size_t need = paged_decode_workspace_size(batch, num_q_heads, pool->num_kv_heads,
                                                    pool->head_dim, pool->block_size,
                                                    static_cast<int32_t>(len), window, prefix);
    if (need > PKV_NO_ALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    // the split partials are written before they are read, so the previous
    // call's contents need no clearing
    return paged_decode_attention(q, num_q_heads, pool, block_tables, max_blocks_per_seq, seq_lens,
                                  batch, max_seq_len, window, scale, out, scratch,
                                  PKV_NO_ALLOC_SCRATCH_BYTES, prefix, dev_status, stream);
}
