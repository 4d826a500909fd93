// Split-KV paged decode over bf16 pools: the launches of the kernel in
// decode_kernel.cuh for each head_dim, one query per row (decode) or a few
// (a speculative-verify step), and of the grouped kernel (several decode
// calls in one launch).
#include "decode_coop.cuh"
#include "decode_kernel.cuh"

namespace pkv {

// A few long rows (the plan's coop flag), one query per row, no shared-prefix
// items and one query n-tile: the cooperative kernel, whose warps share every
// block (decode_coop.cuh).
static bool coop_fits(const DecodeParams &p)
{
    return p.plan.coop && p.cu_q_lens == nullptr && p.plan.n_prefix_ctas == 0 && p.group <= 8 &&
           (p.head_dim == 128 || p.head_dim == 256);
}

cudaError_t launch_decode_bf16(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, cudaStream_t stream)
{
    if (coop_fits(p))
        return p.head_dim == 128 ? launch_coop<128>(p, kmap, vmap, stream)
                                 : launch_coop<256>(p, kmap, vmap, stream);
    const bool mq = p.cu_q_lens != nullptr;  // several queries per row
    // query n-tiles: the rows of a split item (G, or G x max_q for a verify step)
    const bool two = query_ntiles(static_cast<int64_t>(p.group) * (mq ? p.max_q : 1)) == 2;
#define PKV_BF16_LAUNCH(DIM)                                                             \
    return mq ? (two ? launch_split<DIM, true, false, 2>(p, kmap, vmap, stream)           \
                     : launch_split<DIM, true, false, 1>(p, kmap, vmap, stream))          \
              : (two ? launch_split<DIM, false, false, 2>(p, kmap, vmap, stream)          \
                     : launch_split<DIM, false, false, 1>(p, kmap, vmap, stream))
    switch (p.head_dim) {
    case 64: PKV_BF16_LAUNCH(64);
    case 128: PKV_BF16_LAUNCH(128);
    case 256: PKV_BF16_LAUNCH(256);
    default: return cudaErrorInvalidValue;
    }
#undef PKV_BF16_LAUNCH
}

// The groups of one fused call, all on the many-row kernel (the query n-tiles
// follow the group size, which the groups share)
static cudaError_t launch_many_row_grouped(const GroupedDecode &gd, cudaStream_t stream)
{
    const bool two = query_ntiles(gd.g[0].group) == 2;
    switch (gd.g[0].head_dim) {
    case 64: return two ? launch_split_grouped<64, false, 2>(gd, stream) : launch_split_grouped<64, false, 1>(gd, stream);
    case 128: return two ? launch_split_grouped<128, false, 2>(gd, stream) : launch_split_grouped<128, false, 1>(gd, stream);
    case 256: return two ? launch_split_grouped<256, false, 2>(gd, stream) : launch_split_grouped<256, false, 1>(gd, stream);
    default: return cudaErrorInvalidValue;
    }
}

// Every group runs on the kernel its own call would take (each group's
// output equals that call's bit for bit): groups that all take the same
// kernel share one launch; otherwise the cooperative groups and the
// many-row groups get a launch each (one merge launch covers them all).
cudaError_t launch_decode_bf16_grouped(const GroupedDecode &gd, cudaStream_t stream)
{
    GroupedDecode part[2];  // [0]: many-row kernel, [1]: cooperative kernel
    part[0].n = part[1].n = 0;
    int64_t end[2] = {0, 0};
    for (int i = 0; i < gd.n; ++i) {
        const int k = coop_fits(gd.g[i]) ? 1 : 0;
        const int j = part[k].n++;
        part[k].g[j] = gd.g[i];
        part[k].kmap[j] = gd.kmap[i];
        part[k].vmap[j] = gd.vmap[i];
        end[k] += gd.g[i].plan.n_prefix_ctas + gd.g[i].plan.n_suffix_ctas;
        part[k].cta_end[j] = end[k];
    }
    cudaError_t err = cudaSuccess;
    if (part[0].n > 0) err = launch_many_row_grouped(part[0], stream);
    if (err == cudaSuccess && part[1].n > 0)
        err = part[1].g[0].head_dim == 128 ? launch_coop_grouped<128>(part[1], stream)
                                           : launch_coop_grouped<256>(part[1], stream);
    return err;
}

}  // namespace pkv
