// C ABI entry points: argument checks, the split plan, TMA descriptors and
// kernel launches.  Everything here runs on the host; nothing allocates
// device memory and nothing synchronises the stream.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "pkv.h"
#include "pkv_internal.h"


using namespace pkv;

namespace {

std::atomic<int32_t> g_split_override{0};
// diagnostic drill (pkv_set_wait_drill): data-wait limit and flags
std::atomic<uint64_t> g_drill_wait_ns{kWaitLimitNs};
std::atomic<uint32_t> g_drill_flags{0};

// ---------------------------------------------------------------------------
// launch counting and optional per-kind event timing
// ---------------------------------------------------------------------------
std::atomic<int64_t> g_launches{0};
std::atomic<uint32_t> g_prof_mask{0};
struct ProfRecord {
    int kind;
    cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::vector<ProfRecord> g_prof_records;
std::vector<cudaEvent_t> g_prof_free;
cudaEvent_t g_prof_pending[PKV_KERNEL_KINDS] = {};
constexpr size_t kMaxProfRecords = 65536;

cudaEvent_t take_event()
{
    if (!g_prof_free.empty()) {
        cudaEvent_t e = g_prof_free.back();
        g_prof_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

int num_sms_current()
{
    // per-device cache; host threads may call concurrently
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool valid_pool(const pkv_pool *pool)
{
    if (pool == nullptr || pool->k == nullptr || pool->v == nullptr) return false;
    if (pool->num_blocks <= 0 || pool->block_size <= 0 || pool->num_kv_heads <= 0 ||
        pool->head_dim <= 0)
        return false;
    if (pool->dtype != PKV_F32 && pool->dtype != PKV_BF16 && pool->dtype != PKV_FP8_E4M3)
        return false;
    if (pool->dtype == PKV_FP8_E4M3 &&
        (!(std::isfinite(pool->k_scale) && pool->k_scale > 0.f) ||
         !(std::isfinite(pool->v_scale) && pool->v_scale > 0.f)))
        return false;
    return aligned16(pool->k) && aligned16(pool->v);
}

// FP8 pools have one tile layout: 16-token blocks, head_dim a multiple of 64
bool fp8_shape_built(const pkv_pool *pool)
{
    return pool->block_size == 16 &&
           (pool->head_dim == 64 || pool->head_dim == 128 || pool->head_dim == 256);
}

// Element type of queries and outputs: bf16 beside FP8 pools, else the pool's own.
pkv_dtype out_dtype(pkv_dtype t) { return t == PKV_FP8_E4M3 ? PKV_BF16 : t; }

int elem_bytes(pkv_dtype t) { return t == PKV_FP8_E4M3 ? 1 : (t == PKV_BF16 ? 2 : 4); }

// Which decode shapes are built.
bool decode_shape_built(pkv_dtype dtype, int32_t D, int32_t bs, int32_t G)
{
    if (G < 1 || G > 16) return false;
    if (dtype == PKV_BF16 || dtype == PKV_FP8_E4M3)
        return bs == 16 && (D == 64 || D == 128 || D == 256);
    return (D == 32 || D == 64 || D == 128 || D == 256) && bs <= 64 && bs * D <= 4096;
}

// The split plan: a pure function of the sizes and the SM count.
DecodePlan make_plan(int32_t batch, int32_t hq, int32_t hkv, int32_t D, int32_t bs,
                     int32_t max_len, int32_t window, const pkv_prefix_desc *prefix,
                     pkv_dtype dtype, int num_sms)
{
    DecodePlan pl{};
    const int32_t G = hq / hkv;
    int64_t nblk_max = ceil_div64(max_len, bs);
    if (window > 0) nblk_max = std::min<int64_t>(nblk_max, ceil_div64(window, bs) + 1);
    nblk_max = std::max<int64_t>(nblk_max, 1);
    const int64_t tiles_ub = static_cast<int64_t>(batch) * nblk_max * hkv;
    // Split size over the upper bound of (block, kv head) tiles, a multiple of
    // the consumer warp count.  Many (row, kv head) pairs: about nine CTAs
    // per SM (three waves of three resident CTAs), so that rows of unequal
    // length even out, and at least 8 blocks per split (measured on 32 rows of
    // 1-8k tokens: 96 blocks per split beat 64, 72, 80, 108 and 128, for one
    // query per row and for four).  Fewer pairs than SMs (a few long rows):
    // two CTAs per SM, one wave, since each CTA pays a fixed start-up cost
    // and the merge reads every partial; at least 4 blocks per split.
    const int64_t pairs = static_cast<int64_t>(batch) * hkv;
    const bool few = pairs < num_sms;
    const int64_t target = static_cast<int64_t>(std::max(num_sms, 1)) * (few ? 2 : 9);
    int64_t C = ceil_div64(tiles_ub, target);
    C = std::max<int64_t>(C, few ? 4 : 8);
    C = ceil_div64(C, kDecodeWarps) * kDecodeWarps;
    const int32_t ov = g_split_override.load();
    if (ov > 0) C = ov;
    pl.split_blocks = static_cast<int32_t>(C);
    pl.few = few ? 1 : 0;
    pl.n_suffix_splits = static_cast<int32_t>(ceil_div64(nblk_max, C));
    pl.prefix_split_blocks = 8;
    pl.n_prefix_splits = 0;
    pl.prefix_chunks = 0;
    pl.n_prefix_ctas = 0;
    if (prefix != nullptr && prefix->num_groups > 0 && prefix->max_prefix_blocks > 0) {
        // The prefix cut (blocks per prefix split) is sized for a nominal 64
        // (row, head) pairs per CTA (32 at head_dim 256), about one CTA per SM
        // at that size, whatever the dtype, so that the workspace size does
        // not depend on the dtype.  The row chunks then follow the kernel: the
        // bf16 and FP8 kernels take four warp tiles of 8 pairs (G <= 8) or 16
        // per CTA, so at G <= 8 the prefix CTAs come to about two per SM; the
        // f32 kernel takes 16 pairs per CTA.
        const int64_t rows_pairs = static_cast<int64_t>(prefix->max_group_rows) * G;
        const int64_t pairs_bf16 = D == 256 ? kPrefixPairsPerCta / 2 : kPrefixPairsPerCta;
        const int64_t chunks_bf16 = ceil_div64(rows_pairs, pairs_bf16);
        int64_t Cp = ceil_div64(static_cast<int64_t>(prefix->max_prefix_blocks) * hkv *
                                    prefix->num_groups * chunks_bf16,
                                std::max(num_sms, 1));
        Cp = std::min<int64_t>(std::max<int64_t>(Cp, 4), 64);
        int64_t chunks = ceil_div64(rows_pairs, kF32Rows);
        if (dtype != PKV_F32)
            chunks = ceil_div64(rows_pairs, static_cast<int64_t>(kDecodeWarps) * 8 * query_ntiles(G));
        pl.prefix_split_blocks = static_cast<int32_t>(Cp);
        pl.n_prefix_splits = static_cast<int32_t>(ceil_div64(prefix->max_prefix_blocks, Cp));
        pl.prefix_chunks = static_cast<int32_t>(chunks);
        pl.prefix_max = prefix->max_prefix_blocks;
        pl.n_prefix_ctas = static_cast<int64_t>(pl.n_prefix_splits) * hkv * prefix->num_groups * chunks;
    }
    pl.nslot = pl.n_prefix_splits + pl.n_suffix_splits;
    pl.n_suffix_ctas = static_cast<int64_t>(pl.n_suffix_splits) * hkv * batch;
    // The cooperative kernel (its warps share every block) for long runs, or
    // for a grid under half the SMs; runs of 16 blocks over a full grid
    // (4 rows x 2048 tokens) were faster on the many-row kernel (17.4 against
    // 18.9 us per call), runs of 28 (4 rows x 32768) and the 4-block runs of a
    // 512-token window slower (35.9 against 33.4, 15.4 against 12.6 us).
    pl.coop = few && (C >= 24 || 2 * pl.n_suffix_ctas < num_sms) ? 1 : 0;
    return pl;
}

size_t ws_o_bytes(int32_t batch, int32_t hq, int32_t D, const DecodePlan &pl)
{
    const size_t b = static_cast<size_t>(batch) * hq * pl.nslot * D * sizeof(float);
    return (b + 255) & ~static_cast<size_t>(255);
}

size_t ws_total_bytes(int32_t batch, int32_t hq, int32_t D, const DecodePlan &pl)
{
    return ws_o_bytes(batch, hq, D, pl) + static_cast<size_t>(batch) * hq * pl.nslot * 2 * sizeof(float);
}

bool valid_prefix(const pkv_prefix_desc *prefix, int32_t batch, int32_t width)
{
    if (prefix == nullptr || prefix->num_groups == 0) return true;
    if (prefix->num_groups < 0 || prefix->num_groups > batch) return false;
    if (prefix->group_of_row == nullptr || prefix->prefix_blocks == nullptr) return false;
    if (prefix->max_group_rows < 1 || prefix->max_group_rows > batch) return false;
    if (prefix->max_prefix_blocks < 0 || prefix->max_prefix_blocks > width) return false;
    return true;
}

// ---------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn_ready()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 4-D map over a bf16 pool [num_blocks][hkv][bs][D], box 64 dims x bs slots,
// 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, void *base, const pkv_pool &pool)
{
    const cuuint64_t D = pool.head_dim, bs = pool.block_size, hkv = pool.num_kv_heads;
    cuuint64_t dims[4] = {D, bs, hkv, static_cast<cuuint64_t>(pool.num_blocks)};
    cuuint64_t strides[3] = {D * 2, bs * D * 2, hkv * bs * D * 2};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(bs), 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5-D view of the same pool for whole-tile boxes: (64 dims, slot, 64-dim
// region, kv head, block), box (64, bs, D/64, 1, 1).  The region stride (128 B)
// is smaller than the slot stride: the box walks dims, then slots, then
// regions, so a (block, kv head) tile lands region by region, each region
// [bs][64] with the 128-byte swizzle, in one load.
bool encode_pool_map_tile(CUtensorMap *map, void *base, const pkv_pool &pool)
{
    const cuuint64_t D = pool.head_dim, bs = pool.block_size, hkv = pool.num_kv_heads;
    cuuint64_t dims[5] = {64, bs, D / 64, hkv, static_cast<cuuint64_t>(pool.num_blocks)};
    cuuint64_t strides[4] = {D * 2, 128, bs * D * 2, hkv * bs * D * 2};
    cuuint32_t box[5] = {64, static_cast<cuuint32_t>(bs), static_cast<cuuint32_t>(D / 64), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Validation and parameters of one decode call (no launch).  batch == 0
// returns PKV_OK with nothing filled.
pkv_status decode_setup(const void *q, int32_t num_q_heads, const pkv_pool *pool,
                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                        const int32_t *seq_lens, int32_t batch, int32_t max_seq_len,
                        int32_t window, float scale, void *out, void *workspace, size_t ws_bytes,
                        const pkv_prefix_desc *prefix, int32_t *dev_status, DecodeParams *pp)
{
    if (!valid_pool(pool) || batch < 0 || num_q_heads <= 0 || max_seq_len < 0 || window < 0 ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (q == nullptr || out == nullptr || block_tables == nullptr || seq_lens == nullptr ||
        max_blocks_per_seq <= 0 || !aligned16(q) || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    if (!valid_prefix(prefix, batch, max_blocks_per_seq)) return PKV_ERR_INVALID_ARG;
    const bool use_prefix = prefix != nullptr && prefix->num_groups > 0;
    if (use_prefix && window != 0) return PKV_ERR_UNSUPPORTED;
    const int32_t G = num_q_heads / pool->num_kv_heads;
    if (!decode_shape_built(pool->dtype, pool->head_dim, pool->block_size, G))
        return PKV_ERR_UNSUPPORTED;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * pool->block_size;
    const int32_t max_len = static_cast<int32_t>(std::min<int64_t>(max_seq_len, cap));

    const DecodePlan pl = make_plan(batch, num_q_heads, pool->num_kv_heads, pool->head_dim,
                                    pool->block_size, max_len, window,
                                    use_prefix ? prefix : nullptr, pool->dtype, num_sms_current());
    if (pl.n_suffix_ctas > INT32_MAX || pl.n_prefix_ctas > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    const size_t need = ws_total_bytes(batch, num_q_heads, pool->head_dim, pl);
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        ws_bytes < need)
        return PKV_ERR_WORKSPACE;

    DecodeParams &p = *pp;
    p = DecodeParams{};
    p.q = q;
    p.out = out;
    p.k_pool = pool->k;
    p.v_pool = pool->v;
    p.tables = block_tables;
    p.seq_lens = seq_lens;
    p.group_of_row = use_prefix ? prefix->group_of_row : nullptr;
    p.prefix_blocks = use_prefix ? prefix->prefix_blocks : nullptr;
    p.num_groups = use_prefix ? prefix->num_groups : 0;
    p.ws_o = static_cast<float *>(workspace);
    p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                        ws_o_bytes(batch, num_q_heads, pool->head_dim, pl));
    p.status = dev_status;
    p.cu_q_lens = nullptr;  // one query per row
    p.max_q = 1;
    p.batch = batch;
    p.hq = num_q_heads;
    p.hkv = pool->num_kv_heads;
    p.group = G;
    p.head_dim = pool->head_dim;
    p.block_size = pool->block_size;
    p.width = max_blocks_per_seq;
    p.num_blocks = pool->num_blocks;
    p.max_len = max_len;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.v_scale = 1.f;
    if (pool->dtype == PKV_FP8_E4M3) {
        p.scale_log2 *= pool->k_scale;
        p.v_scale = pool->v_scale;
    }
    drill_settings(&p.wait_ns, &p.drill);
    p.plan = pl;
    return PKV_OK;
}

// Groups of one fused call must share what fixes the kernel instantiation.
bool groups_compatible(const pkv_decode_group *groups, int32_t n)
{
    const pkv_pool &p0 = groups[0].pool;
    for (int32_t i = 1; i < n; ++i) {
        const pkv_pool &pi = groups[i].pool;
        if (pi.dtype != p0.dtype || pi.head_dim != p0.head_dim || pi.block_size != p0.block_size ||
            pi.num_kv_heads != p0.num_kv_heads)
            return false;
    }
    return true;
}

}  // namespace

namespace pkv {

void drill_settings(uint64_t *wait_ns, uint32_t *flags)
{
    *wait_ns = g_drill_wait_ns.load();
    *flags = g_drill_flags.load();
}

void prof_begin(int kind, cudaStream_t stream)
{
    g_launches.fetch_add(1);
    if (!(g_prof_mask.load() & (1u << kind))) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_records.size() >= kMaxProfRecords) return;
    cudaEvent_t e = take_event();
    if (e != nullptr && cudaEventRecord(e, stream) == cudaSuccess) g_prof_pending[kind] = e;
}

void prof_end(int kind, cudaStream_t stream)
{
    if (!(g_prof_mask.load() & (1u << kind))) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEvent_t s = g_prof_pending[kind];
    g_prof_pending[kind] = nullptr;
    if (s == nullptr) return;
    cudaEvent_t e = take_event();
    if (e != nullptr && cudaEventRecord(e, stream) == cudaSuccess)
        g_prof_records.push_back({kind, s, e});
    else
        g_prof_free.push_back(s);
}

}  // namespace pkv

extern "C" {

pkv_status pkv_set_wait_drill(uint64_t wait_limit_ns, uint32_t flags)
{
    if ((flags & ~static_cast<uint32_t>(PKV_DRILL_WITHHOLD_FIRST_LOAD)) != 0)
        return PKV_ERR_INVALID_ARG;
    g_drill_wait_ns.store(wait_limit_ns == 0 ? kWaitLimitNs
                                             : std::min<uint64_t>(wait_limit_ns, kWaitLimitNs));
    g_drill_flags.store(flags);
    return PKV_OK;
}

pkv_status pkv_profile_enable(uint32_t kind_mask)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto &r : g_prof_records) {
        g_prof_free.push_back(r.start);
        g_prof_free.push_back(r.stop);
    }
    g_prof_records.clear();
    for (auto &e : g_prof_pending) {
        if (e != nullptr) g_prof_free.push_back(e);
        e = nullptr;
    }
    g_prof_mask.store(kind_mask);
    return PKV_OK;
}

pkv_status pkv_profile_mask(uint32_t kind_mask)
{
    g_prof_mask.store(kind_mask);
    return PKV_OK;
}

pkv_status pkv_profile_read(int32_t kind, int64_t *launches, double *total_ms)
{
    if (kind < 0 || kind >= PKV_KERNEL_KINDS || launches == nullptr || total_ms == nullptr)
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    int64_t n = 0;
    double ms = 0.0;
    for (const auto &r : g_prof_records) {
        if (r.kind != kind) continue;
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            return PKV_ERR_CUDA;
        ++n;
        ms += t;
    }
    *launches = n;
    *total_ms = ms;
    return PKV_OK;
}

pkv_status pkv_profile_times(int32_t kind, float *ms_out, int64_t cap, int64_t *launches)
{
    if (kind < 0 || kind >= PKV_KERNEL_KINDS || launches == nullptr || cap < 0 ||
        (cap > 0 && ms_out == nullptr))
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    int64_t n = 0;
    for (const auto &r : g_prof_records) {
        if (r.kind != kind) continue;
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            return PKV_ERR_CUDA;
        if (n < cap) ms_out[n] = t;
        ++n;
    }
    *launches = n;
    return PKV_OK;
}

int64_t pkv_launch_count(void) { return g_launches.load(); }


const char *pkv_version(void) { return "pkv 0.1 (sm_103a)"; }

const char *pkv_status_string(pkv_status s)
{
    switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported dtype/shape combination";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace too small or misaligned";
    case PKV_ERR_OUT_OF_BLOCKS: return "block pool exhausted at its maximum size";
    }
    return "unknown status";
}

int32_t pkv_set_decode_split_blocks(int32_t blocks_per_split)
{
    return g_split_override.exchange(blocks_per_split > 0 ? blocks_per_split : 0);
}

pkv_status paged_kv_append(const pkv_pool *pool, const int32_t *slot_mapping, int32_t num_tokens,
                           const void *k_new, const void *v_new, int32_t *dev_status,
                           pkv_stream_t stream)
{
    if (!valid_pool(pool) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (slot_mapping == nullptr || k_new == nullptr || v_new == nullptr) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    if (pool->dtype == PKV_FP8_E4M3) {
        if (!fp8_shape_built(pool)) return PKV_ERR_UNSUPPORTED;
        if (static_cast<int64_t>(pool->num_blocks) * pool->block_size > INT32_MAX)
            return PKV_ERR_UNSUPPORTED;
        AppendParams p{};
        p.k_pool = pool->k;
        p.v_pool = pool->v;
        p.k_new = k_new;
        p.v_new = v_new;
        p.slot_mapping = slot_mapping;
        p.status = dev_status;
        p.num_tokens = num_tokens;
        p.hkv = pool->num_kv_heads;
        p.block_size = pool->block_size;
        p.num_slots = pool->num_blocks * pool->block_size;
        p.head_dim = pool->head_dim;
        p.k_scale = pool->k_scale;
        p.v_scale = pool->v_scale;
        return launch_append_fp8(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? PKV_OK
                   : PKV_ERR_CUDA;
    }
    const int64_t row_bytes = static_cast<int64_t>(pool->head_dim) * elem_bytes(pool->dtype);
    if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(pool->num_blocks) * pool->block_size > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    AppendParams p{};
    p.k_pool = pool->k;
    p.v_pool = pool->v;
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.status = dev_status;
    p.num_tokens = num_tokens;
    p.hkv = pool->num_kv_heads;
    p.block_size = pool->block_size;
    p.vecs_per_row = static_cast<int32_t>(row_bytes / 16);
    p.num_slots = pool->num_blocks * pool->block_size;
    return launch_append(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK
                                                                                  : PKV_ERR_CUDA;
}

int32_t pkv_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t max_seq_len, int32_t window,
                        int32_t *blocks_per_split_out)
{
    if (batch < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_seq_len < 0 || window < 0)
        return -1;
    const DecodePlan pl = make_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_seq_len, window, nullptr, PKV_BF16, num_sms_current());
    if (blocks_per_split_out) *blocks_per_split_out = pl.split_blocks;
    return pl.n_suffix_splits;
}

size_t paged_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                   int32_t window, const pkv_prefix_desc *prefix)
{
    if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        head_dim <= 0 || block_size <= 0 || max_seq_len < 0 || window < 0)
        return 0;
    // the f32, bf16 and FP8 plans differ only in how many CTAs cover a
    // prefix group's rows, which does not change the slot count: the size
    // holds for every pool dtype
    const DecodePlan pl = make_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_seq_len, window, prefix, PKV_BF16, num_sms_current());
    return ws_total_bytes(batch, num_q_heads, head_dim, pl);
}

pkv_status paged_decode_attention(const void *q, int32_t num_q_heads, const pkv_pool *pool,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, int32_t batch, int32_t max_seq_len,
                                  int32_t window, float scale, void *out, void *workspace,
                                  size_t ws_bytes, const pkv_prefix_desc *prefix,
                                  int32_t *dev_status, pkv_stream_t stream)
{
    DecodeParams p{};
    const pkv_status stt = decode_setup(q, num_q_heads, pool, block_tables, max_blocks_per_seq,
                                        seq_lens, batch, max_seq_len, window, scale, out,
                                        workspace, ws_bytes, prefix, dev_status, &p);
    if (stt != PKV_OK || batch == 0) return stt;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (pool->dtype == PKV_FP8_E4M3) {
        err = launch_decode_fp8(p, st);
    } else if (pool->dtype == PKV_BF16) {
        if (!encode_fn_ready()) return PKV_ERR_CUDA;
        CUtensorMap kmap, vmap;
        if (!encode_pool_map_tile(&kmap, pool->k, *pool) ||
            !encode_pool_map_tile(&vmap, pool->v, *pool))
            return PKV_ERR_UNSUPPORTED;
        err = launch_decode_bf16(p, kmap, vmap, st);
    } else {
        err = launch_decode_f32(p, st);
    }
    if (err != cudaSuccess) return PKV_ERR_CUDA;
    err = launch_decode_combine(p, out_dtype(pool->dtype), st);
    return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t paged_decode_groups_workspace_size(const pkv_decode_group *groups, int32_t n_groups,
                                          int32_t batch, int32_t num_q_heads)
{
    if (groups == nullptr || n_groups < 1 || n_groups > PKV_MAX_DECODE_GROUPS || batch < 0)
        return 0;
    size_t total = 0;
    for (int32_t i = 0; i < n_groups; ++i) {
        const pkv_decode_group &g = groups[i];
        const size_t one = paged_decode_workspace_size(
            batch, num_q_heads, g.pool.num_kv_heads, g.pool.head_dim, g.pool.block_size,
            g.max_seq_len, g.window, nullptr);
        if (one == 0) return 0;
        total += (one + 255) & ~static_cast<size_t>(255);
    }
    return total;
}

pkv_status paged_decode_attention_groups(const pkv_decode_group *groups, int32_t n_groups,
                                         int32_t batch, int32_t num_q_heads, void *workspace,
                                         size_t ws_bytes, int32_t *dev_status, pkv_stream_t stream)
{
    if (groups == nullptr || n_groups < 1 || n_groups > PKV_MAX_DECODE_GROUPS || batch < 0 ||
        num_q_heads <= 0)
        return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_groups; ++i)
        if (!valid_pool(&groups[i].pool)) return PKV_ERR_INVALID_ARG;
    if (!groups_compatible(groups, n_groups)) return PKV_ERR_INVALID_ARG;
    const pkv_dtype dt = groups[0].pool.dtype;
    if (dt == PKV_F32) return PKV_ERR_UNSUPPORTED;  // the CUDA-core f32 kernel runs per call
    if (batch == 0) return PKV_OK;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        ws_bytes < paged_decode_groups_workspace_size(groups, n_groups, batch, num_q_heads))
        return PKV_ERR_WORKSPACE;
    if (dt == PKV_BF16 && !encode_fn_ready()) return PKV_ERR_CUDA;

    GroupedDecode gd{};
    gd.n = n_groups;
    char *ws = static_cast<char *>(workspace);
    size_t left = ws_bytes;
    int64_t ctas = 0;
    for (int32_t i = 0; i < n_groups; ++i) {
        const pkv_decode_group &g = groups[i];
        const pkv_status stt = decode_setup(g.q, num_q_heads, &g.pool, g.block_tables,
                                            g.max_blocks_per_seq, g.seq_lens, batch, g.max_seq_len,
                                            g.window, g.scale, g.out, ws, left, nullptr,
                                            dev_status, &gd.g[i]);
        if (stt != PKV_OK) return stt;
        const size_t used = (ws_total_bytes(batch, num_q_heads, g.pool.head_dim, gd.g[i].plan) + 255) &
                            ~static_cast<size_t>(255);
        ws += used;
        left -= used;
        ctas += gd.g[i].plan.n_prefix_ctas + gd.g[i].plan.n_suffix_ctas;
        gd.cta_end[i] = ctas;
        if (dt == PKV_BF16 && (!encode_pool_map_tile(&gd.kmap[i], g.pool.k, g.pool) ||
                               !encode_pool_map_tile(&gd.vmap[i], g.pool.v, g.pool)))
            return PKV_ERR_UNSUPPORTED;
    }
    if (ctas > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = dt == PKV_FP8_E4M3 ? launch_decode_fp8_grouped(gd, st)
                                         : launch_decode_bf16_grouped(gd, st);
    if (err != cudaSuccess) return PKV_ERR_CUDA;
    err = launch_decode_combine_grouped(gd, out_dtype(dt), st);
    return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

namespace {

// Chunks whose (query, head) pairs of a kv head fit one 16-row decode tile
// (verify steps of a few queries) run on the split-KV decode kernel.
bool verify_on_decode(int32_t G, int32_t D, int32_t bs, int32_t max_q_len)
{
    return max_q_len >= 1 && static_cast<int64_t>(G) * max_q_len <= 16 &&
           decode_shape_built(PKV_BF16, D, bs, G);
}

// Items of the tensor-core prefill: (row, kv head, query-tile pair).
int32_t prefill_items(int32_t batch, int32_t hq, int32_t hkv, int32_t max_q_len)
{
    if (hkv <= 0 || hq % hkv != 0) return 0;
    const int32_t qpc = prefill_queries_per_cta(PKV_BF16, hq / hkv);
    const int64_t n = static_cast<int64_t>(batch) * hkv * ((max_q_len + qpc - 1) / qpc);
    return n > INT32_MAX ? 0 : static_cast<int32_t>(n);
}

// The decode plan for a verify step: the key range of a row spans its
// queries' windows.
DecodePlan verify_plan(int32_t batch, int32_t hq, int32_t hkv, int32_t D, int32_t bs,
                       int32_t max_len, int32_t window, int32_t max_q_len)
{
    return make_plan(batch, hq, hkv, D, bs, max_len, window > 0 ? window + max_q_len - 1 : 0,
                     nullptr, PKV_BF16, num_sms_current());
}

}  // namespace

extern "C" {

size_t paged_prefill_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int32_t max_q_len,
                                    int32_t max_seq_len, int32_t window)
{
    if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        max_q_len <= 0 || max_seq_len < 0 || window < 0)
        return 0;
    // scratch only for short bf16 chunks: the decode kernel's split partials
    // (a few queries per row), or the prefill kernel's key-range runs
    const int32_t G = num_q_heads / num_kv_heads;
    if (verify_on_decode(G, head_dim, block_size, max_q_len)) {
        const DecodePlan pl = verify_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                          max_seq_len, window, max_q_len);
        return ws_total_bytes(batch * max_q_len, num_q_heads, head_dim, pl);
    }
    const int sms = num_sms_current();
    const PrefillSplit sp = prefill_split_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                               max_q_len, max_seq_len, window, sms);
    const int32_t sk = prefill_sk_ctas(PKV_BF16, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                       max_q_len, sms);
    return std::max(prefill_split_ws_bytes(batch, num_q_heads, max_q_len, sp),
                    prefill_sk_ws_bytes(prefill_items(batch, num_q_heads, num_kv_heads, max_q_len), sk));
}

pkv_status paged_prefill_chunk_attention(const void *q, const int32_t *cu_q_lens,
                                         int32_t num_q_heads, const pkv_pool *pool,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *seq_lens, int32_t batch, int32_t max_q_len,
                                         int32_t max_seq_len, int32_t window, float scale,
                                         void *out, void *workspace, size_t ws_bytes,
                                         int32_t *dev_status, pkv_stream_t stream)
{
    if (!valid_pool(pool) || batch < 0 || num_q_heads <= 0 || max_q_len < 0 || max_seq_len < 0 ||
        window < 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0 || max_q_len == 0) return PKV_OK;
    if (q == nullptr || out == nullptr || cu_q_lens == nullptr || block_tables == nullptr ||
        seq_lens == nullptr || max_blocks_per_seq <= 0 || !aligned16(q) || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    const int32_t G = num_q_heads / pool->num_kv_heads;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * pool->block_size;
    if (pool->dtype != PKV_F32 &&
        verify_on_decode(G, pool->head_dim, pool->block_size, max_q_len)) {
        // a few queries per row: the split-KV decode kernel with (query, head)
        // M-rows, then its merge
        const int32_t max_len = static_cast<int32_t>(std::min<int64_t>(max_seq_len, cap));
        const DecodePlan pl = verify_plan(batch, num_q_heads, pool->num_kv_heads, pool->head_dim,
                                          pool->block_size, max_len, window, max_q_len);
        if (pl.n_suffix_ctas > INT32_MAX) return PKV_ERR_UNSUPPORTED;
        const int32_t prow = batch * max_q_len;
        const size_t need = ws_total_bytes(prow, num_q_heads, pool->head_dim, pl);
        if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
            ws_bytes < need)
            return PKV_ERR_WORKSPACE;
        DecodeParams d{};
        d.q = q;
        d.out = out;
        d.k_pool = pool->k;
        d.v_pool = pool->v;
        d.tables = block_tables;
        d.seq_lens = seq_lens;
        d.group_of_row = nullptr;
        d.prefix_blocks = nullptr;
        d.num_groups = 0;
        d.ws_o = static_cast<float *>(workspace);
        d.ws_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                            ws_o_bytes(prow, num_q_heads, pool->head_dim, pl));
        d.status = dev_status;
        d.cu_q_lens = cu_q_lens;
        d.max_q = max_q_len;
        d.batch = batch;
        d.hq = num_q_heads;
        d.hkv = pool->num_kv_heads;
        d.group = G;
        d.head_dim = pool->head_dim;
        d.block_size = pool->block_size;
        d.width = max_blocks_per_seq;
        d.num_blocks = pool->num_blocks;
        d.max_len = max_len;
        d.window = window;
        d.scale_log2 = scale * 1.4426950408889634f;
        d.v_scale = 1.f;
        drill_settings(&d.wait_ns, &d.drill);
        d.plan = pl;
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        cudaError_t err;
        if (pool->dtype == PKV_FP8_E4M3) {
            d.scale_log2 *= pool->k_scale;
            d.v_scale = pool->v_scale;
            err = launch_decode_fp8(d, st);
        } else {
            if (!encode_fn_ready()) return PKV_ERR_CUDA;
            CUtensorMap kmap, vmap;
            if (!encode_pool_map_tile(&kmap, pool->k, *pool) ||
                !encode_pool_map_tile(&vmap, pool->v, *pool))
                return PKV_ERR_UNSUPPORTED;
            err = launch_decode_bf16(d, kmap, vmap, st);
        }
        if (err == cudaSuccess) err = launch_decode_combine(d, out_dtype(pool->dtype), st);
        return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    }
    if (!prefill_shape_built(pool->dtype, pool->head_dim, pool->block_size, G))
        return PKV_ERR_UNSUPPORTED;
    PrefillParams p{};
    p.q = q;
    p.out = out;
    p.k_pool = pool->k;
    p.v_pool = pool->v;
    p.cu_q_lens = cu_q_lens;
    p.tables = block_tables;
    p.seq_lens = seq_lens;
    p.status = dev_status;
    p.batch = batch;
    p.hq = num_q_heads;
    p.hkv = pool->num_kv_heads;
    p.group = G;
    p.head_dim = pool->head_dim;
    p.block_size = pool->block_size;
    p.width = max_blocks_per_seq;
    p.num_blocks = pool->num_blocks;
    p.max_len = static_cast<int32_t>(std::min<int64_t>(max_seq_len, cap));
    p.max_q_len = max_q_len;
    p.window = window;
    const int32_t qpt = prefill_queries_per_cta(pool->dtype, G);
    p.q_tiles = static_cast<int32_t>(ceil_div64(max_q_len, qpt));
    p.kv_splits = 1;
    p.split_tiles = 0;
    if (pool->dtype != PKV_F32) {
        const PrefillSplit sp = prefill_split_plan(batch, num_q_heads, pool->num_kv_heads,
                                                   pool->head_dim, pool->block_size, max_q_len,
                                                   p.max_len, window, num_sms_current());
        if (sp.splits > 1) {
            const size_t need = prefill_split_ws_bytes(batch, num_q_heads, max_q_len, sp);
            if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                ws_bytes < need)
                return PKV_ERR_WORKSPACE;
            p.kv_splits = sp.splits;
            p.split_tiles = sp.tiles;
            const size_t n = static_cast<size_t>(batch) * max_q_len * num_q_heads * sp.splits;
            p.ws_o = static_cast<float *>(workspace);
            p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                ((n * pool->head_dim * sizeof(float) + 255) &
                                                 ~static_cast<size_t>(255)));
        }
    }
    p.scale_log2 = scale * 1.4426950408889634f;
    p.v_scale = 1.f;
    if (pool->dtype == PKV_FP8_E4M3) {
        p.scale_log2 *= pool->k_scale;
        p.v_scale = pool->v_scale;
    }
    drill_settings(&p.wait_ns, &p.drill);
    p.sk_ctas = 0;
    p.sk_items = 0;
    if (pool->dtype != PKV_F32 && p.kv_splits == 1) {
        const int32_t sk = prefill_sk_ctas(pool->dtype, batch, num_q_heads, pool->num_kv_heads,
                                           pool->head_dim, pool->block_size, max_q_len, num_sms_current());
        if (sk > 0) {
            const int32_t items = prefill_items(batch, num_q_heads, pool->num_kv_heads, max_q_len);
            if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                ws_bytes < prefill_sk_ws_bytes(items, sk))
                return PKV_ERR_WORKSPACE;
            p.sk_ctas = sk;
            p.sk_items = items;
            char *ws = static_cast<char *>(workspace);
            p.sk_prefix = reinterpret_cast<int32_t *>(ws);
            ws += (static_cast<size_t>(items + 1) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
            p.sk_count = reinterpret_cast<int32_t *>(ws);
            ws += (static_cast<size_t>(sk) * 8 * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
            p.sk_o = reinterpret_cast<float *>(ws);
            const size_t rows = static_cast<size_t>(sk) * 2 * 256;
            ws += (rows * 128 * sizeof(float) + 255) & ~static_cast<size_t>(255);
            p.sk_ml = reinterpret_cast<float *>(ws);
        }
    }
    if (static_cast<int64_t>(batch) * p.hkv * p.q_tiles * p.kv_splits > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (pool->dtype == PKV_FP8_E4M3) {
        err = launch_prefill_fp8(p, st);
    } else if (pool->dtype == PKV_BF16) {
        if (!encode_fn_ready()) return PKV_ERR_CUDA;
        CUtensorMap kmap, vmap;
        if (!encode_pool_map(&kmap, pool->k, *pool) || !encode_pool_map(&vmap, pool->v, *pool))
            return PKV_ERR_UNSUPPORTED;
        err = launch_prefill_bf16(p, kmap, vmap, st);
    } else {
        err = launch_prefill_f32(p, st);
    }
    return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"
