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
    // query n-tiles: the rows of a split item (G, or G x max_q for a verify step)
    const bool two = query_ntiles(static_cast<int64_t>(p.group) * (mq ? p.max_q : 1)) == 2;
#define PKV_FP8_LAUNCH(DIM)                                                               \
    return mq ? (two ? launch_split<DIM, true, true, 2>(p, none, none, stream)             \
                     : launch_split<DIM, true, true, 1>(p, none, none, stream))            \
              : (two ? launch_split<DIM, false, true, 2>(p, none, none, stream)            \
                     : launch_split<DIM, false, true, 1>(p, none, none, stream))
    switch (p.head_dim) {
    case 64: PKV_FP8_LAUNCH(64);
    case 128: PKV_FP8_LAUNCH(128);
    case 256: PKV_FP8_LAUNCH(256);
    default: return cudaErrorInvalidValue;
    }
#undef PKV_FP8_LAUNCH
}

cudaError_t launch_decode_fp8_grouped(const GroupedDecode &gd, cudaStream_t stream)
{
    const bool two = query_ntiles(gd.g[0].group) == 2;
    switch (gd.g[0].head_dim) {
    case 64: return two ? launch_split_grouped<64, true, 2>(gd, stream) : launch_split_grouped<64, true, 1>(gd, stream);
    case 128: return two ? launch_split_grouped<128, true, 2>(gd, stream) : launch_split_grouped<128, true, 1>(gd, stream);
    case 256: return two ? launch_split_grouped<256, true, 2>(gd, stream) : launch_split_grouped<256, true, 1>(gd, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
