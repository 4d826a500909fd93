// Split-KV paged decode over bf16 pools: the launches of the kernel in
// decode_kernel.cuh for each head_dim, one query per row (decode) or a few
// (a speculative-verify step), and of the grouped kernel (several decode
// calls in one launch).
#include "decode_kernel.cuh"

namespace pkv {

cudaError_t launch_decode_bf16(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, cudaStream_t stream)
{
    const bool mq = p.cu_q_lens != nullptr;  // several queries per row
    switch (p.head_dim) {
    case 64: return mq ? launch_split<64, true, false>(p, kmap, vmap, stream)
                       : launch_split<64, false, false>(p, kmap, vmap, stream);
    case 128: return mq ? launch_split<128, true, false>(p, kmap, vmap, stream)
                        : launch_split<128, false, false>(p, kmap, vmap, stream);
    case 256: return mq ? launch_split<256, true, false>(p, kmap, vmap, stream)
                        : launch_split<256, false, false>(p, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_bf16_grouped(const GroupedDecode &gd, cudaStream_t stream)
{
    switch (gd.g[0].head_dim) {
    case 64: return launch_split_grouped<64, false>(gd, stream);
    case 128: return launch_split_grouped<128, false>(gd, stream);
    case 256: return launch_split_grouped<256, false>(gd, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
