// Internal host/device interface between the C ABI layer (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pkv.h"

namespace pkv {

// Upper bound on any pipeline wait; a wait that runs past it reports
// PKV_DEV_TIMEOUT and the kernel winds down instead of spinning on.  The
// kernels' data waits take their limit from the launch parameters (this value
// unless a diagnostic drill shortens it); the waits of a wind-down, for copies
// a CTA issued itself, always take this one.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Diagnostic drill flag carried by the launch parameters (pkv_set_wait_drill):
// the first load of every pipeline is never issued, so that the wait for it
// runs out with nothing in flight on its barrier.
constexpr uint32_t kDrillWithholdFirst = PKV_DRILL_WITHHOLD_FIRST_LOAD;

struct AppendParams {
    void *k_pool;
    void *v_pool;
    const void *k_new;
    const void *v_new;
    const int32_t *slot_mapping;
    int32_t *status;
    int32_t num_tokens;
    int32_t hkv;
    int32_t block_size;
    int32_t vecs_per_row;  // head_dim * elem_bytes / 16 (bf16/f32 pools)
    int32_t num_slots;     // num_blocks * block_size
    int32_t head_dim;      // FP8 pools: bf16 rows are quantized with these scales
    float k_scale, v_scale;
    int32_t heads_per_warp;  // FP8: kv heads one warp quantizes for a token (divides hkv)
};

// Split plan of one decode call.  A row's key range [lo, L) covers the blocks
// b_first .. b_end-1; split s of the row's suffix covers blocks
// b_first + s*split_blocks .. (capped at b_end).  Rows of a shared-prefix
// group start their suffix at the group's prefix_blocks, and the prefix is cut
// into runs of prefix_split_blocks read once for the whole group.
struct DecodePlan {
    int32_t split_blocks;         // C
    int32_t n_suffix_splits;      // splits per row (upper bound)
    int32_t prefix_split_blocks;  // Cp
    int32_t n_prefix_splits;      // prefix splits per group (upper bound); 0 = no prefix path
    int32_t nslot;                // partial slots per (row, q head) = n_prefix + n_suffix
    int32_t prefix_chunks;        // CTAs per (group, kv head, prefix split) over its rows
    int32_t prefix_max;           // prefix lengths are clamped to this (<= table width)
    int32_t few;                  // rows x kv heads < SMs: a few long rows, about two CTAs per SM
    int32_t coop;                 // few, and runs long enough (or a grid small enough) for the
                                  // cooperative kernel (bf16, one query per row, G <= 8)
    int64_t n_prefix_ctas;
    int64_t n_suffix_ctas;
};

struct DecodeParams {
    const void *q;
    void *out;
    const void *k_pool;  // read directly by the f32 and FP8 kernels; bf16 goes through TMA maps
    const void *v_pool;
    const int32_t *tables;
    const int32_t *seq_lens;
    const int32_t *group_of_row;   // nullptr when there is no prefix path
    const int32_t *prefix_blocks;
    float *ws_o;   // [batch * max_q][hq][nslot][head_dim] unnormalised weighted values
    float *ws_ml;  // [batch * max_q][hq][nslot][2]: running max (log2 units) and weight sum
    int32_t *status;
    // several queries per row (a speculative-verify step; bf16 only): row r
    // owns the packed queries cu_q_lens[r] .. cu_q_lens[r+1]-1 at the last
    // positions of its length, causally.  nullptr: one query per row (decode)
    const int32_t *cu_q_lens;
    int32_t max_q;  // queries per row, upper bound (1 for decode)
    int32_t batch, hq, hkv, group, head_dim, block_size, width, num_blocks;
    int32_t max_len;   // min(max_seq_len, width * block_size): lengths are clamped to it
    int32_t window;
    int32_t num_groups;
    float scale_log2;  // scale * log2(e) (* k_scale for FP8): scores are kept in base-2 units
    float v_scale;     // FP8: applied to each partial's weighted values
    uint64_t wait_ns;  // limit of the pipeline's data waits (kWaitLimitNs unless a drill)
    uint32_t drill;    // diagnostic drill flags (kDrillWithholdFirst); 0 normally
    DecodePlan plan;
};

// Several decode calls fused into one split launch and one merge launch.
constexpr int kMaxDecodeGroups = 4;
struct GroupedDecode {
    CUtensorMap kmap[kMaxDecodeGroups];  // bf16 pools (unused for FP8)
    CUtensorMap vmap[kMaxDecodeGroups];
    DecodeParams g[kMaxDecodeGroups];
    int64_t cta_end[kMaxDecodeGroups];   // split CTAs of groups 0..i (cumulative)
    int64_t item_end[kMaxDecodeGroups];  // merge CTAs of groups 0..i (cumulative)
    int32_t n;
};

// Launch with programmatic stream serialization (PDL): the kernel may be
// scheduled while the previous kernel on the stream drains; it calls
// pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch bookkeeping (api.cu): every kernel launch is counted; launches of
// kinds enabled by pkv_profile_enable are bracketed by CUDA events.
void prof_begin(int kind, cudaStream_t stream);
void prof_end(int kind, cudaStream_t stream);

struct PrefillParams {
    const void *q;
    void *out;
    const void *k_pool;  // used by the f32 kernel; the bf16 kernel reads via TMA
    const void *v_pool;
    const int32_t *cu_q_lens;
    const int32_t *tables;
    const int32_t *seq_lens;
    int32_t *status;
    int32_t batch, hq, hkv, group, head_dim, block_size, width, num_blocks;
    int32_t max_len;    // min(max_seq_len, width * block_size)
    int32_t max_q_len;
    int32_t window;
    int32_t q_tiles;    // CTAs per (row, kv head): ceil(max_q_len / queries per CTA)
    // key-range split (bf16, short chunks only; 1 = none): each (row, kv head,
    // query tile) is cut into kv_splits runs of split_tiles 64-key tiles whose
    // fp32 partials a merge kernel combines
    int32_t kv_splits;
    int32_t split_tiles;
    float *ws_o;   // [batch][max_q_len][hq][kv_splits][128] unnormalised weighted values
    float *ws_ml;  // [batch][max_q_len][hq][kv_splits][2]: reference max (log2 units), weight sum
    // persistent balanced schedule ("stream-K"; 0 = off): sk_ctas CTAs take
    // equal runs of the (item, 64-key tile) sequence of the sk_items items
    // (row, kv head, query-tile pair); a run that cuts an item writes a
    // partial to one of its CTA's two slots
    int32_t sk_ctas, sk_items;
    int32_t *sk_prefix;  // [sk_items + 1]: tiles of items 0 .. u-1 (written by the plan kernel)
    int32_t *sk_count;   // [sk_ctas][2 query tiles][4 warps]: pieces done of the item cut
                         // after the CTA's first tile (zeroed by the plan kernel)
    float *sk_o;         // [sk_ctas][2][256 rows][128] unnormalised weighted values
    float *sk_ml;        // [sk_ctas][2][256 rows][2]: reference max (log2 units), weight sum
    float scale_log2;  // scale * log2(e) (* k_scale for FP8 pools)
    float v_scale;     // FP8 pools: applied to the weighted values
    uint64_t wait_ns;  // limit of the pipeline's data waits (kWaitLimitNs unless a drill)
    uint32_t drill;    // diagnostic drill flags (kDrillWithholdFirst); 0 normally
};

// The current diagnostic drill (pkv_set_wait_drill): the data-wait limit and
// the flags every decode / prefill launch carries.
void drill_settings(uint64_t *wait_ns, uint32_t *flags);

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_append_fp8(const AppendParams &p, cudaStream_t stream);
bool prefill_shape_built(pkv_dtype dtype, int32_t D, int32_t bs, int32_t G);
int32_t prefill_queries_per_cta(pkv_dtype dtype, int32_t G);
// Key-range split of the bf16 prefill for short chunks (all of a row's
// queries in one query tile) on grids too small to fill the GPU: runs per
// (row, kv head) and 64-key tiles per run; {1, 0} = no split.
struct PrefillSplit {
    int32_t splits, tiles;
};
PrefillSplit prefill_split_plan(int32_t batch, int32_t hq, int32_t hkv, int32_t D, int32_t bs,
                                int32_t max_q_len, int32_t max_seq_len, int32_t window,
                                int num_sms);
size_t prefill_split_ws_bytes(int32_t batch, int32_t hq, int32_t max_q_len, const PrefillSplit &sp);
// The persistent balanced schedule of the tensor-core prefill: the CTA count
// (0 = off: the grid then holds one CTA per item) and its workspace.
int32_t prefill_sk_ctas(pkv_dtype dtype, int32_t batch, int32_t hq, int32_t hkv, int32_t D,
                        int32_t bs, int32_t max_q_len, int num_sms);
size_t prefill_sk_ws_bytes(int32_t items, int32_t ctas);
cudaError_t launch_prefill_bf16(const PrefillParams &p, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, cudaStream_t stream);
cudaError_t launch_prefill_f32(const PrefillParams &p, cudaStream_t stream);
cudaError_t launch_prefill_fp8(const PrefillParams &p, cudaStream_t stream);

// bf16 pools: TMA + mbarrier pipeline, mma.sync tiles.  kmap/vmap: 5-D tensor
// maps (64 dims, slot, 64-dim region, kv head, block), whole-tile boxes, 128B swizzle.
cudaError_t launch_decode_bf16(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, cudaStream_t stream);
// f32 pools: CUDA-core kernel.
cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_decode_fp8(const DecodeParams &p, cudaStream_t stream);
// grouped launches (decode only: one query per row, no prefix path); the
// merge covers every group with the same kernel shape
cudaError_t launch_decode_bf16_grouped(const GroupedDecode &gd, cudaStream_t stream);
cudaError_t launch_decode_fp8_grouped(const GroupedDecode &gd, cudaStream_t stream);
cudaError_t launch_decode_combine_grouped(GroupedDecode &gd, pkv_dtype out_dtype, cudaStream_t stream);
// merge of the split partials into out (dtype of q)
cudaError_t launch_decode_combine(const DecodeParams &p, pkv_dtype dtype, cudaStream_t stream);

// Warps per decode CTA: a split CTA's warps share one query tile and take its
// blocks in turn; a shared-prefix CTA holds one tile of (row, head) pairs per
// warp.  The prefix cut (the prefix blocks per split) is sized as if a CTA
// held 64 pairs (32 at head_dim 256), whatever the dtype, so that the
// workspace size does not depend on it.
constexpr int kDecodeWarps = 4;
constexpr int kPrefixPairsPerCta = 64;  // head_dim <= 128 (32 for head_dim 256)

// bf16 / FP8 decode: query rows sit on the N side of the products in n-tiles
// of 8; a split item's rows (the G heads, or G x queries of a verify step)
// need this many, and so does each warp's tile of a prefix item (8 x that
// many (row, head) pairs per warp)
inline int query_ntiles(int64_t rows) { return rows > 8 ? 2 : 1; }
// query rows per CTA of the f32 kernel
constexpr int kF32Rows = 16;

}  // namespace pkv
