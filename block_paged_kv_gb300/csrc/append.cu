// Append of new K/V rows into their pool slots ("perf.md", paged knob table:
// the graph-native paged K/V write, MLX_PAGED_NATIVE_KV_WRITE).
//
// One thread moves one 16-byte vector of one (token, kv head) row for both K
// and V: two 16-byte loads and two 16-byte stores, all coalesced within the
// row (a bf16 head_dim-128 row is 16 vectors).  HBM bound: the algorithmic
// traffic is 2 x (read + write) x num_tokens x Hkv x head_dim x elem bytes plus
// 4 bytes of slot per token.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int VPT>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p)
{
    // vector v of row (t, h):  idx = (t * hkv + h) * vecs_per_row + v
    pdl_wait();
    pdl_trigger();
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.hkv * p.vecs_per_row;
    // each block covers VPT * blockDim consecutive vectors, one warp-wide
    // contiguous run per unrolled step
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int64_t idx =
            (static_cast<int64_t>(blockIdx.x) * VPT + u) * blockDim.x + threadIdx.x;
        if (idx >= total) return;
        const int32_t v = static_cast<int32_t>(idx % p.vecs_per_row);
        const int64_t th = idx / p.vecs_per_row;
        const int32_t h = static_cast<int32_t>(th % p.hkv);
        const int32_t t = static_cast<int32_t>(th / p.hkv);
        const int32_t slot = __ldg(p.slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (h == 0 && v == 0) report(p.status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int32_t blk = slot / p.block_size;
        const int32_t off = slot - blk * p.block_size;
        const int64_t dst = ((static_cast<int64_t>(blk) * p.hkv + h) * p.block_size + off) *
                                p.vecs_per_row + v;
        const uint4 kv = __ldcs(reinterpret_cast<const uint4 *>(p.k_new) + idx);
        const uint4 vv = __ldcs(reinterpret_cast<const uint4 *>(p.v_new) + idx);
        reinterpret_cast<uint4 *>(p.k_pool)[dst] = kv;
        reinterpret_cast<uint4 *>(p.v_pool)[dst] = vv;
    }
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.hkv * p.vecs_per_row;
    if (total == 0) return cudaSuccess;
    constexpr int kVpt = 2;
    const int64_t blocks = (total + kVpt * 256 - 1) / (kVpt * 256);
    prof_begin(PKV_KERNEL_APPEND, stream);
    const cudaError_t err = launch_pdl(append_kernel<kVpt>, dim3(static_cast<unsigned>(blocks)),
                                       dim3(256), 0, stream, p);
    prof_end(PKV_KERNEL_APPEND, stream);
    return err;
}

}  // namespace pkv
