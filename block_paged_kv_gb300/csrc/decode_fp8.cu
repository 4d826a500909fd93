// Split-KV paged decode over FP8 (E4M3) pools ("perf.md", quantisation scheme
// table: the paged adapter's FP8 KV cache with per-layer scales): the launches
// of the kernel in decode_kernel.cuh for each head_dim.  Tiles come in by bulk
// copy from the pool pointers, so no tensor maps are needed.
#include "decode_kernel.cuh"

namespace pkv {

cudaError_t launch_decode_fp8(const DecodeParams &p, cudaStream_t stream)
{
    const CUtensorMap none{};  // unused by the FP8 instantiations
    const bool mq = p.cu_q_lens != nullptr;
    switch (p.head_dim) {
    case 64: return mq ? launch_split<64, true, true>(p, none, none, stream)
                       : launch_split<64, false, true>(p, none, none, stream);
    case 128: return mq ? launch_split<128, true, true>(p, none, none, stream)
                        : launch_split<128, false, true>(p, none, none, stream);
    case 256: return mq ? launch_split<256, true, true>(p, none, none, stream)
                        : launch_split<256, false, true>(p, none, none, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
