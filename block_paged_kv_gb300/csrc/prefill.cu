// Chunked prefill against a paged prefix ("perf.md", gather_kv_for_prefill_chunk:
// a prefill chunk attends its cached prefix through the pages; "paged-cache.md":
// chunk boundaries change the reduction order, not the result).  Query i of a
// row's chunk sits at absolute position p = L - C + i and attends positions
// max(0, p - W + 1) .. p: the whole prefix and the chunk causally.
//
// Tensor-core kernel (bf16 pools; FP8 pools the same kernel with widening),
// work item = (row, kv head, two tiles of 128/G queries).  A tile's 128 M-rows
// are (query, head) pairs of all G q heads of the kv head, and both tiles
// share every K/V tile, so K/V are loaded once per 256 query rows.  QK^T and
// PV are dense contractions and run on the 5th-generation tensor cores:
//   warps 0/2 producers: K and V tiles of 64 keys (4 paged blocks) into
//             4-stage rings (bf16: two 64-dim TMA boxes a block; FP8: bulk
//             copies of the E4M3 blocks into a two-deep staging buffer); a K
//             stage is freed once both S products are computed and the key
//             masks read, a V stage once both P.V products are;
//   warps 1/3 issue tile A's / tile B's tcgen05.mma from one elected lane:
//             S = Q K^T into one of the tile's two S buffers in tensor memory
//             (both operands K-major, 128-byte swizzle), O += P V with P read
//             from tensor memory; per K/V tile j, once K(j+2) has landed and
//             P(j) is stored: P(j).V, then S(j+2) into the buffer that product
//             reads.  Warp 1 also allocates the 512 tensor-memory columns;
//   warps 4-7 / 8-11  softmax of tile A / tile B, concurrently, one M-row per
//             thread: S from tensor memory, causal / window / range mask,
//             running max kept within 2^8 of the true maximum (O is rescaled
//             in tensor memory only when it moves further), P written back
//             over S (bf16: hi + lo terms, 8 columns each per 16 keys, so
//             that P.V carries P to ~2^-17 relative; FP8 pools: one f16
//             term), and the epilogue O / l.  FP8 pools: tile A's warps also
//             widen the staged K tiles to f16, tile B's the V tiles.
// Schedules: one CTA per item while the items fit one wave; more items than
// SMs: one persistent CTA per SM (a whole item, then an equal run of the
// remaining items' tiles, cut pieces merged in the kernel).  A short chunk
// fills tile A only (tile B's warps stay idle, warps whose rows hold no query
// skip the softmax work); on a grid too small for the GPU its key range is
// cut into runs whose fp32 partials prefill_merge_kernel merges.
// f32 kernel: CUDA cores, the same work split with 16 (query, head) pairs per
// CTA, for the fp32 pools.
#include <algorithm>

#include "decode_common.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace pf {
constexpr int kD = 128;
constexpr int kRows = 128;                // M of one query tile
constexpr int kQTiles = 2;                // query tiles per CTA, sharing every K/V tile
constexpr int kKeys = 64;                 // keys per K/V tile (4 blocks of 16)
constexpr int kBlocks = kKeys / 16;
constexpr int kQBytes = kRows * 2 * 128;  // one query tile: two 64-dim swizzled regions
constexpr int kKVRegion = kKeys * 128;    // 8 KiB: one 64-dim half of a K/V tile
constexpr int kTileBytes = 2 * kKVRegion; // 16 KiB: a K or a V tile
constexpr int kStages = 4;                // K ring and V ring depth
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQTiles * kQBytes;
constexpr int kVOff = kKOff + kStages * kTileBytes;
// FP8 pools: the producers stage each tile's E4M3 bytes (4 blocks x 2 KiB)
// by bulk copy, two tiles deep, and widen them into the ring
constexpr int kF8BlockBytes = 16 * kD;                 // one (block, kv head) E4M3 tile
constexpr int kF8StageTile = kBlocks * kF8BlockBytes;  // 8 KiB
constexpr int kSoftmaxWarps = 8;  // 4-7 softmax of query tile A, 8-11 of tile B
template <bool kF8>
struct Layout {
    static constexpr int kStagingOff = kVOff + kStages * kTileBytes;
    static constexpr int kStagingBytes = kF8 ? 2 * 2 * kF8StageTile : 0;  // K and V, 2 deep
    static constexpr int kBarOff = kStagingOff + kStagingBytes;
    // barriers: k_full[4], k_empty[4], v_full[4], v_empty[4], s_full[tile][buf],
    // p_full[tile][buf], pv_done[tile], mma_drain[tile], q_full[tile],
    // FP8: staged[K/V][2], stg_free[K/V][2]
    static constexpr int kNumBars = 4 * kStages + 4 + 4 + 2 + 2 + 2 + (kF8 ? 8 : 0);
    // kmask[kStages], FP8: smask[K/V][2] (blocks loaded of each staging buffer)
    static constexpr int kMaskOff = kBarOff + kNumBars * 8;
    static constexpr int kTmemOff = kMaskOff + (kStages + 4) * 4;
    static constexpr int kSegOff = kTmemOff + 16;  // per softmax warp: its segment walk
    static constexpr int kBytes = kSegOff + kSoftmaxWarps * 96;
    static constexpr int kLaunchBytes = kBytes + 1024;
    static_assert(kLaunchBytes <= 227 * 1024, "shared memory of one CTA");
};
// warps: 0 K producer, 1 MMA issue for tile A, 2 V producer, 3 MMA issue for
// tile B;
// 4-7 softmax of query tile A, 8-11 of tile B (one M-row per thread)
constexpr int kThreads = 384;
// tensor memory: S_x[buf] (64 columns each) at 128x + 64buf, O_x at 256 + 128x
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRescaleLog2 = 8;      // O is rescaled only when the max grows past 2^8
}  // namespace pf

struct PrefillRowInfo {
    int32_t r, g, i0, nq, L, C, kv_lo, kv_hi, s;
};

__device__ __forceinline__ bool prefill_item(const PrefillParams &p, int64_t bid, int qpc,
                                             PrefillRowInfo &w)
{
    w.s = static_cast<int32_t>(bid % p.kv_splits);
    bid /= p.kv_splits;
    const int32_t qt = static_cast<int32_t>(bid % p.q_tiles);
    bid /= p.q_tiles;
    w.g = static_cast<int32_t>(bid % p.hkv);
    w.r = static_cast<int32_t>(bid / p.hkv);
    const int32_t c0 = __ldg(p.cu_q_lens + w.r), c1 = __ldg(p.cu_q_lens + w.r + 1);
    int32_t C = c1 - c0;
    int32_t L = __ldg(p.seq_lens + w.r);
    const bool report_bad = qt == 0 && w.g == 0;
    if (L < 0 || L > p.max_len) {
        if (report_bad) report(p.status, PKV_DEV_BAD_LEN);
        L = L < 0 ? 0 : p.max_len;
    }
    if (c0 < 0 || C < 0 || C > p.max_q_len || C > L) {
        if (report_bad) report(p.status, PKV_DEV_BAD_LEN);
        C = c0 < 0 || C < 0 ? 0 : min(min(C, p.max_q_len), L);
    }
    w.C = C;
    w.L = L;
    w.i0 = qt * qpc;
    if (w.i0 >= C) return false;
    w.nq = min(qpc, C - w.i0);
    const int32_t p_first = L - C + w.i0;
    w.kv_hi = p_first + w.nq;
    w.kv_lo = p.window > 0 ? max(0, p_first - p.window + 1) : 0;
    return true;
}

// Wait by every lane of the warp (false in all lanes if any gave up); reports
// a timeout.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int lane, int32_t *status,
                                          unsigned long long limit_ns)
{
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns));
    if (!ok && lane == 0) report(status, PKV_DEV_TIMEOUT);
    return ok;
}

// ---------------------------------------------------------------------------
// Segments: the (item, key-tile range) pieces a CTA works through.  An item
// is a (row, kv head, query-tile pair); its key tiles are the 64-key tiles of
// its key range [kv_lo, kv_hi).
//   one CTA per item (sk_ctas == 0): one segment, the item's whole range or,
//     for the key-range runs of a short chunk, one run of it;
//   persistent balanced schedule (sk_ctas = n > 0, fewer than the items):
//     the items' tiles in item order form one sequence of W tiles
//     (sk_prefix, written by prefill_sk_plan_kernel).  CTA c first runs item
//     c whole (the CTAs of one (row, kv head) then start together and share
//     its K/V through L2), then takes the tiles [B + c R / n, B + (c + 1) R
//     / n) of the rest (B = the first n items' tiles, R = W - B), item by
//     item.  Only the first and the last segment of that run can cut an
//     item; a cut segment writes a partial to slot 0 (first) or 1 (last) of
//     the CTA, and the warp that completes an item's pieces merges them.
// ---------------------------------------------------------------------------
struct Seg {
    PrefillRowInfo w;
    int32_t item;
    int32_t jt0;    // first key tile of the segment (in 64-key units)
    int32_t ntile;  // tiles of the segment
    bool whole;     // the item's whole key range
    int32_t slot;   // persistent schedule: partial slot of a cut segment
};

struct SegWalk {
    int32_t pos, end;  // persistent schedule: tiles of the CTA's run still ahead
    int32_t u;         // the item holding tile pos
    int32_t k;         // segments returned so far
};

// start of CTA c's balanced run (c = n: the end of the sequence)
__device__ __forceinline__ int32_t sk_run_start(const PrefillParams &p, int32_t c)
{
    const int64_t B = __ldg(p.sk_prefix + p.sk_ctas), W = __ldg(p.sk_prefix + p.sk_items);
    return static_cast<int32_t>(B + static_cast<int64_t>(c) * (W - B) / p.sk_ctas);
}

// the item holding tile pos: the largest u with prefix[u] <= pos
__device__ __forceinline__ int32_t sk_item_of(const PrefillParams &p, int32_t pos)
{
    int32_t lo = 0, hi = p.sk_items;
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (__ldg(p.sk_prefix + mid) <= pos) lo = mid; else hi = mid;
    }
    return lo;
}

// the CTA whose balanced run holds tile pos (pos past the first n items)
__device__ __forceinline__ int32_t sk_cta_of(const PrefillParams &p, int32_t pos)
{
    const int64_t B = __ldg(p.sk_prefix + p.sk_ctas), W = __ldg(p.sk_prefix + p.sk_items);
    int32_t c = W > B ? static_cast<int32_t>((pos - B) * static_cast<int64_t>(p.sk_ctas) / (W - B)) : 0;
    c = min(max(c, 0), p.sk_ctas - 1);
    while (c + 1 < p.sk_ctas && sk_run_start(p, c + 1) <= pos) ++c;
    while (c > 0 && sk_run_start(p, c) > pos) --c;
    return c;
}

// Next segment of a persistent CTA's run (false at its end).
__device__ __forceinline__ bool sk_next(const PrefillParams &p, int qpc, SegWalk &sw, Seg &sg)
{
    if (sw.pos >= sw.end) return false;
    const int32_t u = sw.u;
    const int32_t lo = __ldg(p.sk_prefix + u), hi = __ldg(p.sk_prefix + u + 1);
    const int32_t seg_end = min(hi, sw.end);
    prefill_item(p, u, qpc, sg.w);  // an item with tiles has queries
    sg.item = u;
    sg.jt0 = sg.w.kv_lo / pf::kKeys + (sw.pos - lo);
    sg.ntile = seg_end - sw.pos;
    sg.whole = sw.pos == lo && seg_end == hi;
    sg.slot = sw.k == 0 ? 0 : 1;
    ++sw.k;
    sw.pos = seg_end;
    if (seg_end == hi) {
        int32_t v = u + 1;  // skip items without tiles (no queries)
        while (v < p.sk_items && __ldg(p.sk_prefix + v + 1) == __ldg(p.sk_prefix + v)) ++v;
        sw.u = v;
    }
    return true;
}

// First segment of CTA `cta` (false: nothing to do).  One CTA per item: the
// item (or its key-range run; an empty run sets ntile <= 0).
__device__ __forceinline__ bool seg_first(const PrefillParams &p, int qpc, int64_t cta, SegWalk &sw,
                                          Seg &sg)
{
    if (p.sk_ctas > 0) {
        const int32_t c = static_cast<int32_t>(cta);
        sw.pos = sk_run_start(p, c);
        sw.end = sk_run_start(p, c + 1);
        sw.k = 0;
        sw.u = sw.pos < sw.end ? sk_item_of(p, sw.pos) : 0;
        const int32_t lo = __ldg(p.sk_prefix + c), hi = __ldg(p.sk_prefix + c + 1);
        if (hi > lo) {  // item c, whole
            prefill_item(p, c, qpc, sg.w);  // an item with tiles has queries
            sg.item = c;
            sg.jt0 = sg.w.kv_lo / pf::kKeys;
            sg.ntile = hi - lo;
            sg.whole = true;
            sg.slot = 0;
            return true;
        }
        return sk_next(p, qpc, sw, sg);
    }
    if (!prefill_item(p, cta, qpc, sg.w)) return false;
    sg.item = static_cast<int32_t>(cta);
    sg.jt0 = sg.w.kv_lo / pf::kKeys;
    sg.ntile = (sg.w.kv_hi - 1) / pf::kKeys - sg.jt0 + 1;
    sg.whole = p.kv_splits <= 1;
    sg.slot = 0;
    if (!sg.whole) {
        const int32_t tb = sg.w.s * p.split_tiles;
        sg.ntile = min(sg.ntile, tb + p.split_tiles) - tb;
        sg.jt0 += tb;
    }
    sw.pos = sw.end = 0;  // no further segment
    return true;
}

__device__ __forceinline__ bool seg_next(const PrefillParams &p, int qpc, SegWalk &sw, Seg &sg)
{
    return p.sk_ctas > 0 && sk_next(p, qpc, sw, sg);
}

// The key tiles of a CTA in order, over its segments (producers).
struct TileCursor {
    SegWalk sw;
    Seg sg;
    int32_t j;  // tile within the segment
    bool valid;
    __device__ __forceinline__ void start(const PrefillParams &p, int qpc, const SegWalk &w0, const Seg &s0)
    {
        sw = w0;
        sg = s0;
        j = 0;
        valid = s0.ntile > 0;
        (void)p;
        (void)qpc;
    }
    __device__ __forceinline__ void advance(const PrefillParams &p, int qpc)
    {
        if (!valid) return;
        if (++j < sg.ntile) return;
        j = 0;
        valid = seg_next(p, qpc, sw, sg);
    }
    __device__ __forceinline__ int32_t kt() const { return sg.jt0 + j; }  // absolute key tile
};

// One row of a query tile into shared memory (softmax thread ii = 0 .. 255:
// tile ii / 128, row i = ii % 128 = (query x*qpt + i/G, head i%G)), 128-byte
// swizzled for the tensor cores.  FP8 pools take f16 products (bf16 -> f16 is
// exact inside the f16 range; a magnitude past 65504 sets PKV_DEV_Q_RANGE); a
// negative scale is staged as -q (`flip` toggles the sign bits), so that the
// scores the tensor cores produce always take a positive factor.  Not inlined:
// a segment's staging then leaves the registers of the softmax loop around
// it alone.
template <bool kF8>
__device__ __noinline__ void stage_q_row(const uint4 *q, const int32_t *cu_q_lens, int32_t hq, int G,
                                         int qpt, int32_t r, int32_t i0, int32_t nq, int32_t g,
                                         uint32_t flip, int32_t *status, uint8_t *q_s, int ii)
{
    constexpr int kD = pf::kD, kRows = pf::kRows;
    const int x = ii / kRows, i = ii % kRows;
    const int t = x * qpt + i / G, h = i % G;
    const bool valid = i < qpt * G && t < nq;
    const uint4 *src = q + ((static_cast<int64_t>(__ldg(cu_q_lens + r)) + i0 + t) * hq + g * G + h) * (kD / 8);
    uint8_t *qt_s = q_s + x * pf::kQBytes;
    bool qbad = false;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        if constexpr (kF8) {
            v.x = bf16x2_to_f16x2(v.x, qbad);
            v.y = bf16x2_to_f16x2(v.y, qbad);
            v.z = bf16x2_to_f16x2(v.z, qbad);
            v.w = bf16x2_to_f16x2(v.w, qbad);
        }
        v.x ^= flip;
        v.y ^= flip;
        v.z ^= flip;
        v.w ^= flip;
        *reinterpret_cast<uint4 *>(qt_s + (c >> 3) * (kRows * 128) + i * 128 + (((c & 7) ^ (i & 7)) << 4)) = v;
    }
    if (qbad) report(status, PKV_DEV_Q_RANGE);
    fence_proxy_async_smem();  // read by the tensor cores (async proxy)
}

// ---------------------------------------------------------------------------
// bf16, tcgen05
// ---------------------------------------------------------------------------
template <bool kF8>
__global__ void __launch_bounds__(pf::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PrefillParams p)
{
    using namespace pf;
    using L = Layout<kF8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *q_s = smem + kQOff;
    uint8_t *k_s = smem + kKOff;
    uint8_t *v_s = smem + kVOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *k_full = bars, *k_empty = bars + kStages, *v_full = bars + 2 * kStages,
             *v_empty = bars + 3 * kStages;
    uint64_t *s_full = bars + 4 * kStages;      // [tile * 2 + buf]
    uint64_t *p_full = bars + 4 * kStages + 4;  // [tile * 2 + buf]
    uint64_t *pv_done = bars + 4 * kStages + 8; // [tile]
    uint64_t *mma_drain = bars + 4 * kStages + 10;  // [tile]: the issuer's last products
    uint64_t *q_full = bars + 4 * kStages + 12;     // [tile]: a segment's query tile staged
    uint64_t *staged = bars + 4 * kStages + 14;  // FP8: [K/V * 2 + buffer]
    uint64_t *stg_free = bars + 4 * kStages + 18;  // FP8: [K/V * 2 + buffer] widened by the softmax warps
    uint32_t *kmask = reinterpret_cast<uint32_t *>(smem + L::kMaskOff);
    uint32_t *smask = kmask + kStages;  // FP8: [K/V * 2 + buffer] blocks loaded of a staging buffer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kTmemOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int qpt = kRows / G;  // queries per query tile

    if (!kF8 && threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    pdl_wait();
    pdl_trigger();

    const int qpc = kQTiles * qpt;  // queries per item
    SegWalk sw0;
    Seg seg0;
    if (!seg_first(p, qpc, blockIdx.x, sw0, seg0)) return;
    const bool split = p.kv_splits > 1;  // one CTA per key-range run of a short chunk
    if (split && seg0.ntile <= 0) {
        // an empty run: an empty partial (no weight) for every live row
        const PrefillRowInfo &w = seg0.w;
        if (warp >= 4) {
            const int x = (warp >> 2) - 1, row = 32 * (warp & 3) + lane;
            const int t = x * qpt + row / G;
            if (row < qpt * G && t < w.nq) {
                const size_t pi = ((static_cast<size_t>(w.r) * p.max_q_len + w.i0 + t) * p.hq +
                                   w.g * G + row % G) * p.kv_splits + w.s;
                *reinterpret_cast<float2 *>(p.ws_ml + pi * 2) = make_float2(-INFINITY, 0.f);
            }
        }
        return;
    }
    // query tiles with queries in them: a short chunk (a verify step of a few
    // queries) fills tile A only, and tile B's warps then stay idle; the
    // persistent schedule runs both (its segments' items differ)
    const int nqt = (p.sk_ctas > 0 || seg0.w.nq > qpt) ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            // the S products of the live tiles + their warpgroups' kmask reads
            mbar_init(&k_empty[i], nqt + nqt * (kSoftmaxWarps / kQTiles));
            // FP8: one softmax warpgroup widens K into the stages, the other
            // V (tile A's both when it runs alone); bf16: one TMA arrival
            mbar_init(&k_full[i], kF8 ? kSoftmaxWarps / kQTiles : 1);
            mbar_init(&v_full[i], kF8 ? kSoftmaxWarps / kQTiles : 1);
            mbar_init(&v_empty[i], nqt);  // the live tiles' P.V products
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kSoftmaxWarps / kQTiles);
        }
        mbar_init(&pv_done[0], 1);
        mbar_init(&pv_done[1], 1);
        mbar_init(&mma_drain[0], 1);
        mbar_init(&mma_drain[1], 1);
        mbar_init(&q_full[0], kSoftmaxWarps / kQTiles);
        mbar_init(&q_full[1], kSoftmaxWarps / kQTiles);
        if (kF8) {
            for (int i = 0; i < 4; ++i) mbar_init(&staged[i], 1);
            for (int i = 0; i < 4; ++i) mbar_init(&stg_free[i], kSoftmaxWarps / kQTiles);
        }
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(tmem_slot, kTmemCols);

    // query tiles: tile x row i = (query t = x * qpt + i / G, head h = i % G);
    // the 256 softmax threads load one row each (the first segment's here,
    // the next segments' after each epilogue)
    // a negative scale: stage -q (sign bits flipped, exact), so that the
    // scores the tensor cores produce always take a positive factor
    const uint32_t flip = p.scale_log2 < 0.f ? 0x80008000u : 0u;
    auto load_q_row = [&](const PrefillRowInfo &w) {
        stage_q_row<kF8>(static_cast<const uint4 *>(p.q), p.cu_q_lens, p.hq, G, qpt, w.r, w.i0, w.nq,
                         w.g, flip, p.status, q_s, threadIdx.x - 128);
    };
    if (warp >= 4) load_q_row(seg0.w);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tS = [&](int x, int buf) { return tmem + 128u * static_cast<uint32_t>(x) + 64u * static_cast<uint32_t>(buf); };
    auto tO = [&](int x) { return tmem + 256u + 128u * static_cast<uint32_t>(x); };

    if (warp == 0 || warp == 2) {
        // ------------------------------------------ K (warp 0) / V (warp 2) producer
        // The CTA's key tiles in order over its segments; tile T (a running
        // count) goes to ring stage T % kStages.
        const bool is_k = warp == 0;
        // diagnostic drill: tile 0's loads are never issued (its waits run out)
        auto withheld = [&](int32_t T) { return (p.drill & kDrillWithholdFirst) != 0 && T == 0; };
        uint8_t *ring = is_k ? k_s : v_s;
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *empty = is_k ? k_empty : v_empty;
        // lane < kBlocks: logical block kt * kBlocks + lane of the cursor's
        // tile, inside the table and the item's key range
        auto in_range_of = [&](const TileCursor &c) {
            const int32_t kb = c.kt() * kBlocks + lane;
            return c.valid && lane < kBlocks && kb < p.width && kb * 16 < c.sg.w.kv_hi &&
                   (kb + 1) * 16 > c.sg.w.kv_lo;
        };
        auto load_id = [&](const TileCursor &c) {
            return in_range_of(c) ? __ldg(p.tables + static_cast<int64_t>(c.sg.w.r) * p.width +
                                          c.kt() * kBlocks + lane)
                                  : -1;
        };
        if constexpr (kF8) {
            // FP8: tile T's E4M3 blocks are bulk-copied into staging buffer
            // T % 2 (two tiles ahead of the ring), then widened to f16 into
            // the ring stage: K as the bf16 path lays it out (key rows, 64-dim
            // 128-byte-swizzled regions), V transposed (dim rows of the tile's
            // 64 keys, 128-byte swizzled), so that a pair of codes becomes
            // one 4-byte store.  Value columns of keys outside [kv_lo, kv_hi)
            // or of blocks not loaded are written as zeros (stale slots may
            // hold NaN codes).
            const uint64_t policy = l2_evict_last_policy();  // re-read by the row's other CTAs
            const uint8_t *pool = static_cast<const uint8_t *>(is_k ? p.k_pool : p.v_pool);
            uint8_t *stg = smem + L::kStagingOff + (is_k ? 0 : 2) * kF8StageTile;
            uint64_t *stg_bar = staged + (is_k ? 0 : 2);
            int32_t nf = 0;  // tiles 0 .. nf-1 fetched into the staging buffers
            // fetch tile nf at cursor c (block ids read one tile before);
            // whole warp; returns the mask of loaded blocks
            auto fetch = [&](const TileCursor &c, int32_t id) {
                const bool in_range = in_range_of(c);
                const bool good = in_range && static_cast<uint32_t>(id) < static_cast<uint32_t>(p.num_blocks);
                if (is_k && in_range && !good) report(p.status, PKV_DEV_BAD_BLOCK);
                const uint32_t mask = __ballot_sync(0xffffffffu, good) & ((1u << kBlocks) - 1u);
                const int32_t tile = nf++;
                const int sb = tile & 1;
                if (lane == 0) smask[(is_k ? 0 : 2) + sb] = mask;  // published by the arrival below
                if (withheld(tile)) return mask;  // diagnostic drill: never issued
                if (lane == 0) {
                    if (mask == 0)
                        mbar_arrive(&stg_bar[sb]);
                    else
                        mbar_arrive_expect_tx(&stg_bar[sb], __popc(mask) * kF8BlockBytes);
                }
                __syncwarp();
#pragma unroll
                for (int b = 0; b < kBlocks; ++b) {
                    const int32_t bid = __shfl_sync(0xffffffffu, id, b);
                    if (((mask >> b) & 1u) && elect_one())
                        bulk_load(stg + sb * kF8StageTile + b * kF8BlockBytes,
                                  pool + (static_cast<int64_t>(bid) * p.hkv + c.sg.w.g) * kF8BlockBytes,
                                  kF8BlockBytes, &stg_bar[sb], policy);
                }
                __syncwarp();
                return mask;
            };
            // bulk copies only, two tiles ahead; the softmax warps widen each
            // tile into the ring and release the staging buffer
            TileCursor cf, ci;
            cf.start(p, qpc, sw0, seg0);
            ci = cf;
            int32_t id_next = load_id(ci);
            ci.advance(p, qpc);
            int32_t T = 0;
            for (; cf.valid; ++T, cf.advance(p, qpc)) {
                const int sb = T & 1;
                if (T >= 2 && !warp_wait(&stg_free[(is_k ? 0 : 2) + sb], ((T >> 1) + 1) & 1, lane, p.status,
                                         p.wait_ns))
                    break;
                fetch(cf, id_next);
                id_next = load_id(ci);
                ci.advance(p, qpc);
            }
            // the copies this warp issued have landed before it leaves
            if (lane == 0)
                for (int32_t t = max(0, T - 2); t < T; ++t)
                    if (!withheld(t)) mbar_wait(&stg_bar[t & 1], (t >> 1) & 1);
            __syncwarp();
        } else {
            const CUtensorMap *map = is_k ? &kmap : &vmap;
            const uint64_t policy = l2_evict_last_policy();  // re-read by the row's other CTAs
            TileCursor cur;
            cur.start(p, qpc, sw0, seg0);
            int32_t T = 0;
            for (; cur.valid; ++T, cur.advance(p, qpc)) {
                const int st = T % kStages;
                if (T >= kStages && !warp_wait(&empty[st], ((T / kStages) + 1) & 1, lane, p.status, p.wait_ns)) break;
                const bool in_range = in_range_of(cur);
                const int32_t id = load_id(cur);
                const bool good = in_range && static_cast<uint32_t>(id) < static_cast<uint32_t>(p.num_blocks);
                if (is_k && in_range && !good) report(p.status, PKV_DEV_BAD_BLOCK);
                const uint32_t mask = __ballot_sync(0xffffffffu, good) & ((1u << kBlocks) - 1u);
                if (is_k && lane == 0) kmask[st] = mask;
                if (withheld(T)) continue;  // diagnostic drill: never issued
                if (lane == 0) {
                    if (mask == 0)
                        mbar_arrive(&full[st]);
                    else
                        mbar_arrive_expect_tx(&full[st], __popc(mask) * 2 * 2048);
                }
                __syncwarp();
                uint8_t *dst = ring + st * kTileBytes;
                const int32_t g = cur.sg.w.g;
#pragma unroll
                for (int b = 0; b < kBlocks; ++b) {
                    const int32_t bid = __shfl_sync(0xffffffffu, id, b);
                    if (((mask >> b) & 1u) && elect_one()) {
                        tma_load_4d(dst + b * 2048, map, &full[st], 0, 0, g, bid, policy);
                        tma_load_4d(dst + kKVRegion + b * 2048, map, &full[st], 64, 0, g, bid, policy);
                    }
                }
            }
            // wind-down (a wait ran out) and normal exit alike: the loads of
            // the last ring's worth of tiles have landed before the warp
            // leaves (at a normal exit their consumers saw them land already)
            if (lane == 0)
                for (int32_t t = max(0, T - kStages); t < T; ++t)
                    if (!withheld(t)) mbar_wait(&full[t % kStages], (t / kStages) & 1);
            __syncwarp();
        }
    } else if (warp == 1 || (warp == 3 && nqt == 2)) {
        // ------------------------------------------------------------ MMA issue
        // Warp 1 issues tile A's products, warp 3 tile B's.  Per K/V tile j:
        // P(j).V, then S(j+2) = Q K(j+2)^T into the S buffer that product just
        // read.  With two S buffers a warpgroup finds S(j+1) computed when it
        // finishes P(j).  One thread's products execute in issue order, so a
        // product never overtakes an earlier read of the same columns.
        const int x = warp >> 1;
        // bf16: V is MN-major (key rows); FP8: V^T is K-major (dim rows of keys)
        constexpr uint32_t idS = kF8 ? tc::idesc_f16(kRows, kKeys, 0, 0) : tc::idesc_bf16(kRows, kKeys, 0, 0);
        constexpr uint32_t idO = kF8 ? tc::idesc_f16(kRows, kD, 0, 0) : tc::idesc_bf16(kRows, kD, 0, 1);
        // Descriptors are built once; moving along K (or to the next 16 keys
        // of V) adds the byte offset / 16 to the start-address field, which
        // cannot carry out of it inside shared memory.
        const uint64_t dq = tc::smem_desc(smem_u32(q_s + x * kQBytes), 16, 1024);
        const uint64_t dk = tc::smem_desc(smem_u32(k_s), 16, 1024);
        const uint64_t dv = kF8 ? tc::smem_desc(smem_u32(v_s), 16, 1024)
                                : tc::smem_desc(smem_u32(v_s), kKVRegion, 1024);
        // the B operand of the keys 16kk .. 16kk+15: bf16 key rows 16kk.. (2 KiB
        // on); FP8 32 bytes along each dim row
        constexpr uint64_t kVStep = kF8 ? (32 >> 4) : (2048 >> 4);
        constexpr uint64_t kStageStep = kTileBytes >> 4;
        const uint32_t tO_x = tO(x);
        // The whole warp waits; one elected lane issues a step's products and
        // commits from one straight-line block.
        auto k_landed = [&](int32_t T) {  // K(T) landed (T: the CTA's running tile count)
            return warp_wait(&k_full[T % kStages], (T / kStages) & 1, lane, p.status, p.wait_ns);
        };
        auto s_issue = [&](int32_t T) {  // S(T) = Q K(T)^T
            const uint64_t kd = dk + static_cast<uint64_t>(T % kStages) * kStageStep;
            const uint32_t d = tS(x, T & 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t qo = static_cast<uint64_t>(((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4);
                const uint64_t ko = static_cast<uint64_t>(((kk >> 2) * kKVRegion + (kk & 3) * 32) >> 4);
                tc::mma_ss(d, dq + qo, kd + ko, idS, kk > 0 ? 1u : 0u);
            }
            tc::commit(&s_full[x * 2 + (T & 1)]);
            tc::commit(&k_empty[T % kStages]);
        };
        // O += P(T) V(T); V(T) has landed (the warpgroup checked it before
        // handing P over); a segment's first tile starts O afresh
        auto pv_issue = [&](int32_t T, bool seg_start) {
            const uint64_t vd = dv + static_cast<uint64_t>(T % kStages) * kStageStep;
            const uint32_t a = tS(x, T & 1);
            const uint32_t first = seg_start ? 0u : 1u;
            // bf16: keys 16g..16g+15 hold P hi in S columns 16g..16g+7 and P
            // lo in 16g+8..16g+15 (bf16 pairs); FP8 pools: one f16 term, keys
            // 16g..16g+15 in columns 8g..8g+7
#pragma unroll
            for (int part = 0; part < (kF8 ? 1 : 2); ++part)
#pragma unroll
                for (int kk = 0; kk < kBlocks; ++kk)
                    tc::mma_ts(tO_x, a + (kF8 ? 8 : 16) * kk + 8 * part, vd + kVStep * static_cast<uint64_t>(kk),
                               idO, (part > 0 || kk > 0) ? 1u : first);
            tc::commit(&pv_done[x]);
            tc::commit(&v_empty[T % kStages]);
        };
        SegWalk sw = sw0;
        Seg sg = seg0;
        int32_t T0 = 0;  // the segment's first tile in the running count
        for (int32_t k = 0;; ++k) {
            const int32_t n = sg.ntile;
            // the segment's query tile is staged (the previous segment's
            // products, which read the old one, completed before its epilogue)
            bool ok = warp_wait(&q_full[x], k & 1, lane, p.status, p.wait_ns);
            ok = ok && k_landed(T0) && (n < 2 || k_landed(T0 + 1));
            if (ok) {
                tc::fence_after();
                if (elect_one()) {
                    s_issue(T0);
                    if (n >= 2) s_issue(T0 + 1);
                }
                __syncwarp();
            }
            // per tile: K(T+2) is waited for first (it landed, or was widened,
            // long before P(T) is ready), so that P(T).V(T) and S(T+2) leave
            // in one block as soon as P(T) is
            for (int32_t j = 0; j < n && ok; ++j) {
                const int32_t T = T0 + j;
                const bool more = j + 2 < n;
                if (more) ok = k_landed(T + 2);
                ok = ok && warp_wait(&p_full[x * 2 + (T & 1)], (T >> 1) & 1, lane, p.status, p.wait_ns);
                if (!ok) break;
                tc::fence_after();
                if (elect_one()) {
                    pv_issue(T, j == 0);
                    if (more) s_issue(T + 2);
                }
                __syncwarp();
            }
            if (!ok) break;
            T0 += n;
            if (!seg_next(p, qpc, sw, sg)) break;
        }
        // every product this warp issued has completed before the CTA frees
        // tensor memory (after a wait ran out, some may still be running)
        if (elect_one()) tc::commit(&mma_drain[x]);
        __syncwarp();
        mbar_wait(&mma_drain[x], 0);
        __syncwarp();
    } else if (warp >= 4 && (warp < 8 || nqt == 2)) {
        // ------------------------------------------------------------ softmax
        // warpgroup x (warps 4-7: tile A, 8-11: tile B), one M-row per thread:
        // tensor-memory lane quarter warp % 4, the 64 key columns of S
        const int x = (warp >> 2) - 1;
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const int row = 32 * (warp & 3) + lane;
        const int t = x * qpt + row / G;
        const uint32_t ox = tO(x) + lane_base;
        // |scale| * log2(e) (q was staged negated for a negative scale), kept
        // away from 0 so that a masked score (-inf) never meets a zero factor
        const float sl = fmaxf(fabsf(p.scale_log2), 1e-30f);
        bool abort = false;
        // FP8: tile A's warpgroup widens K, tile B's V (tile A's both when it
        // runs alone), each 128 threads over a tile's 512 staged chunks: a
        // warp then waits for one staging and one ring barrier per tile, and
        // the two warpgroups need not run in step.
        // K(Tk)'s staged E4M3 chunks, this thread's share, widened to f16
        // into ring stage Tk % kStages (key rows, 64-dim 128-byte-swizzled
        // regions, as the bf16 path lays them out); keys of blocks not loaded
        // are left as they are (their scores are masked).  The stage is free
        // once tile Tk - kStages's S products and mask reads are done.
        const int nthr = kRows;
        const bool do_k = nqt == 1 || x == 0, do_v = nqt == 1 || x == 1;
        const int wq0 = (threadIdx.x - 128) & (kRows - 1);  // this thread's first chunk
        auto widen_k = [&](int32_t Tk) {
            const int sb = Tk & 1, st = Tk % kStages;
            bool okw = mbar_wait(&staged[sb], (Tk >> 1) & 1, p.wait_ns);
            if (Tk >= kStages) okw = okw && mbar_wait(&k_empty[st], ((Tk / kStages) + 1) & 1, p.wait_ns);
            if (__any_sync(0xffffffffu, !okw)) return false;
            const uint32_t km = smask[sb];
            if (threadIdx.x == 128) kmask[st] = km;  // for the score masks of tile Tk
            const uint32_t src = smem_u32(smem + L::kStagingOff + sb * kF8StageTile);
            const uint32_t dst = smem_u32(k_s + st * kTileBytes);
            // A warp takes 32 chunks of one (block, 64-dim group, token half):
            // lane l holds key 8 half + l/4, dims 16kk + 2(l%4) + {0, 1, 8, 9}
            // (kk = 0..3), i.e. the 8x8 matrices (keys) x (dims 16kk + 8h ..
            // + 7) in the fragment order that stmatrix stores as 16-byte rows.
            // Matrix 2kk + h is 16-byte chunk 2kk + h of each key's 128-byte
            // row, swizzled by the key row.
            const int mr = lane & 7, mm = lane >> 3;  // this lane's row address: row mr of matrix mm
            for (int q = wq0; q < kBlocks * 128; q += nthr) {
                const int b = q >> 7, ch = q & 127;  // warp-uniform but for ch % 32
                if (!((km >> b) & 1u)) continue;
                const int grp = ch >> 6, half = (ch >> 5) & 1;
                const uint4 q4 = lds128(src + b * kF8BlockBytes + ch * 16);
                uint32_t f[8];  // f[2kk + h]: matrix (kk, h)
                e4m3x4_to_f16x2x2(q4.x, f[0], f[1]);
                e4m3x4_to_f16x2x2(q4.y, f[2], f[3]);
                e4m3x4_to_f16x2x2(q4.z, f[4], f[5]);
                e4m3x4_to_f16x2x2(q4.w, f[6], f[7]);
                const int krow = b * 16 + half * 8 + mr;
                const uint32_t rowa = dst + grp * kKVRegion + krow * 128;
                stsm_x4(rowa + ((mm ^ mr) << 4), f[0], f[1], f[2], f[3]);
                stsm_x4(rowa + (((4 + mm) ^ mr) << 4), f[4], f[5], f[6], f[7]);
            }
            // read by the tensor cores (async proxy); the staging buffer is
            // refilled by bulk copies after these generic-proxy reads
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&k_full[st]);
                mbar_arrive(&stg_free[sb]);
            }
            return true;
        };
        // the CTA's tiles over all its segments
        const int32_t T_total =
            p.sk_ctas > 0 ? __ldg(p.sk_prefix + blockIdx.x + 1) - __ldg(p.sk_prefix + blockIdx.x) +
                                sk_run_start(p, blockIdx.x + 1) - sk_run_start(p, blockIdx.x)
                          : seg0.ntile;
        if constexpr (kF8) {
            for (int32_t Tk = 0; do_k && Tk < min(2, T_total) && !abort; ++Tk)
                if (!widen_k(Tk)) {
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                    abort = true;
                }
        }
        // this warp's segment walk and current segment live in shared memory
        // (lane 0 writes them): the tile loop keeps its registers
        struct SegSmem {
            SegWalk sw;
            Seg sg;
        };
        static_assert(sizeof(SegSmem) <= 96, "the per-warp segment slot");
        SegSmem *ss = reinterpret_cast<SegSmem *>(smem + L::kSegOff) + (warp - 4);
        if (lane == 0) {
            ss->sw = sw0;
            ss->sg = seg0;
        }
        __syncwarp();
        int32_t T0 = 0;  // the segment's first tile in the running count
        for (int32_t k = 0; !abort; ++k) {
        const int32_t ntile = ss->sg.ntile, jt0 = ss->sg.jt0;
        const int32_t kv_lo = ss->sg.w.kv_lo, kv_hi = ss->sg.w.kv_hi;
        // the segment's query tile: staged (the first in the prologue), then
        // handed to the MMA-issue warp
        if (k > 0) load_q_row(ss->sg.w);
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[x]);
        const bool valid_row = row < qpt * G && t < ss->sg.w.nq;
        const int32_t qpos = ss->sg.w.L - ss->sg.w.C + ss->sg.w.i0 + t;
        const int32_t qlo = p.window > 0 ? max(0, qpos - p.window + 1) : 0;
        float m_ref = -INFINITY, l = 0.f;
        const bool warp_live = __any_sync(0xffffffffu, valid_row);
        for (int32_t jj = 0; jj < ntile; ++jj) {
            const int32_t T = T0 + jj;
            const int ks = T % kStages, buf = T & 1;
            const int32_t tbase = (jt0 + jj) * kKeys;
            const uint32_t sx = tS(x, buf) + lane_base;
            if constexpr (kF8) {
                if (do_k && T + 2 < T_total && !widen_k(T + 2)) {
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                    abort = true;
                    break;
                }
            }
            if (kF8 && do_v) {
                // V(T): this thread's share of the staged E4M3 chunks widened to
                // f16 into ring stage T % kStages, transposed (dim rows of the
                // tile's 64 keys, 128-byte swizzled); value columns of keys
                // outside [kv_lo, kv_hi) or of blocks not loaded as zeros.  The
                // stage is free once both tiles' P.V(T - kStages) completed.
                const int sb = T & 1;
                bool okw = mbar_wait(&staged[2 + sb], (T >> 1) & 1, p.wait_ns);
                if (T >= kStages) okw = okw && mbar_wait(&v_empty[ks], ((T / kStages) + 1) & 1, p.wait_ns);
                if (__any_sync(0xffffffffu, !okw)) {
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                    abort = true;
                    break;
                }
                const uint32_t vm = smask[2 + sb];
                const uint32_t src = smem_u32(smem + L::kStagingOff + 2 * kF8StageTile + sb * kF8StageTile);
                const uint32_t dst = smem_u32(v_s + ks * kTileBytes);
                const bool vedge = tbase < kv_lo || tbase + kKeys > kv_hi;
                // A warp takes the 32 chunks of one (block, 32-dim group): lane
                // l holds dim 32g + 8jn + l/4 (jn = 0..3) for keys 16b + 2(l%4)
                // + {0, 1, 8, 9}, i.e. the 8x8 matrices (dims 32g + 8jn .. + 7)
                // x (keys 16b + 8h .. + 7) in stmatrix fragment order.  Matrix
                // (jn, h) is 16-byte chunk 2b + h of each dim row, swizzled by
                // the dim row.
                const int mr = lane & 7, mm = lane >> 3, c = lane & 3;
                for (int q = wq0; q < kBlocks * 128; q += nthr) {
                    const int b = q >> 7, ch = q & 127;  // warp-uniform but for ch % 32
                    const int g32 = ch >> 5;
                    uint32_t f[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // f[2jn + h]: matrix (jn, h)
                    if ((vm >> b) & 1u) {
                        const uint4 q4 = lds128(src + b * kF8BlockBytes + ch * 16);
                        e4m3x4_to_f16x2x2(q4.x, f[0], f[1]);
                        e4m3x4_to_f16x2x2(q4.y, f[2], f[3]);
                        e4m3x4_to_f16x2x2(q4.z, f[4], f[5]);
                        e4m3x4_to_f16x2x2(q4.w, f[6], f[7]);
                        if (vedge) {
                            auto live = [&](int k) {
                                const int32_t kp = tbase + b * 16 + k;
                                return kp >= kv_lo && kp < kv_hi;
                            };
                            const uint32_t mk0 = (live(2 * c) ? 0x0000ffffu : 0u) | (live(2 * c + 1) ? 0xffff0000u : 0u);
                            const uint32_t mk1 = (live(2 * c + 8) ? 0x0000ffffu : 0u) | (live(2 * c + 9) ? 0xffff0000u : 0u);
#pragma unroll
                            for (int jn = 0; jn < 4; ++jn) {
                                f[2 * jn] &= mk0;
                                f[2 * jn + 1] &= mk1;
                            }
                        }
                    }
                    // row mr of matrix mm: dim 32g + 8(jn0 + mm/2) + mr, chunk 2b + mm%2
                    const uint32_t rowa = dst + (g32 * 32 + (mm >> 1) * 8 + mr) * 128;
                    const uint32_t cx = static_cast<uint32_t>(((2 * b + (mm & 1)) ^ mr) << 4);
                    stsm_x4(rowa + cx, f[0], f[1], f[2], f[3]);
                    stsm_x4(rowa + 16 * 128 + cx, f[4], f[5], f[6], f[7]);
                }
                // read by the tensor cores (async proxy); the staging buffer is
                // refilled by bulk copies after these generic-proxy reads
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&v_full[ks]);
                    mbar_arrive(&stg_free[2 + sb]);
                }
            }
            bool got = mbar_wait(&s_full[x * 2 + buf], (T >> 1) & 1, p.wait_ns);
            got = got && mbar_wait(&k_full[ks], (T / kStages) & 1, p.wait_ns);  // for kmask
            if (__any_sync(0xffffffffu, !got)) {
                if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                abort = true;
                break;
            }
            const uint32_t mask = kmask[ks];
            __syncwarp();
            if (lane == 0) mbar_arrive(&k_empty[ks]);
            tc::fence_after();
            // a warp whose 32 rows hold no query (a short chunk fills only the
            // first rows of the tile) leaves its S rows alone: the P.V product
            // then writes only O rows that are never stored
            if (warp_live) {
                float s[64];
                {
                    uint32_t r0[32], r1[32];
                    tc::ld32(sx, r0);
                    tc::ld32(sx + 32, r1);
                    tc::wait_ld();
    #pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        s[e] = __uint_as_float(r0[e]);
                        s[32 + e] = __uint_as_float(r1[e]);
                    }
                }
                // a tile with any key outside this row's range takes the masked
                // path: key column e is attended iff e - lo is in [0, qpos - qlo]
                // and its block was loaded
                const bool full = mask == (1u << kBlocks) - 1u && tbase >= qlo &&
                                  tbase + kKeys - 1 <= qpos && valid_row;
                if (!full) {
                    const int32_t lo = qlo - tbase;
                    const uint32_t span = static_cast<uint32_t>(qpos - qlo);  // qlo <= qpos
                    const uint32_t bm = valid_row ? mask : 0u;
    #pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const bool ok = static_cast<uint32_t>(e - lo) <= span && ((bm >> (e >> 4)) & 1u);
                        s[e] = ok ? s[e] : -INFINITY;
                    }
                }
                float mt;
                {
                    float m8[8];
    #pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        m8[e] = fmax3(s[e], s[8 + e], s[16 + e]);
                        m8[e] = fmax3(m8[e], s[24 + e], s[32 + e]);
                        m8[e] = fmax3(m8[e], s[40 + e], s[48 + e]);
                        m8[e] = fmaxf(m8[e], s[56 + e]);
                    }
                    mt = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], fmax3(m8[5], m8[6], m8[7]))) * sl;
                }
                // keep the reference max within 2^8 of the running max
                const float new_ref = (mt > m_ref + static_cast<float>(kRescaleLog2)) ? mt : m_ref;
                const float alpha = fast_exp2(m_ref - new_ref);  // 0 from -inf, 1 if unchanged
                const bool resc = new_ref != m_ref && m_ref != -INFINITY;
                if (__any_sync(0xffffffffu, resc)) {
                    // O_x holds P.V up to tile jj-1 once that product completes
                    if (jj > 0) {
                        const bool done = mbar_wait(&pv_done[x], (T - 1) & 1, p.wait_ns);
                        if (__any_sync(0xffffffffu, !done)) {
                            if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                            abort = true;
                            break;
                        }
                        tc::fence_after();
                    }
                    const float f = resc ? alpha : 1.f;
    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r32[32];
                        tc::ld32(ox + c * 32, r32);
                        tc::wait_ld();
    #pragma unroll
                        for (int e = 0; e < 32; ++e) r32[e] = __float_as_uint(__uint_as_float(r32[e]) * f);
                        tc::st32(ox + c * 32, r32);
                    }
                    tc::wait_st();
                }
                m_ref = new_ref;
                const float nmu = new_ref == -INFINITY ? 0.f : -new_ref;
                // key pairs in paired fp32 arithmetic: 2^(s * sl - m), the
                // row sum in two paired accumulators
                const uint64_t sl2 = f2_pack(sl, sl), nmu2 = f2_pack(nmu, nmu);
                uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
                auto p_pair = [&](int k, float &a, float &b) {
                    f2_unpack(f2_fma(f2_pack(s[k], s[k + 1]), sl2, nmu2), a, b);
                    a = fast_exp2(a);
                    b = fast_exp2(b);
                };
                if constexpr (kF8) {
                    // one f16 term: keys 2c, 2c+1 -> column c, in place
    #pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[16];
    #pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float a, b;
                            p_pair(32 * h + 2 * e, a, b);
                            ls2[e & 1] = f2_add(ls2[e & 1], f2_pack(a, b));
                            pk[e] = pack_f16x2(a, b);
                        }
                        tc::st16(sx + 16 * h, pk);
                    }
                } else {
                    // group g (16 keys) -> 8 columns of P hi then 8 of P lo
    #pragma unroll
                    for (int g = 0; g < kBlocks; ++g) {
                        uint32_t pk[16];
    #pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float a, b;
                            p_pair(16 * g + 2 * e, a, b);
                            const uint64_t ab = f2_pack(a, b);
                            ls2[e & 1] = f2_add(ls2[e & 1], ab);
                            const uint32_t hi = pack_bf16x2(a, b);
                            pk[e] = hi;
                            float ra, rb;
                            f2_unpack(f2_sub(ab, f2_pack(bf16lo_to_f32(hi), bf16hi_to_f32(hi))), ra, rb);
                            pk[8 + e] = pack_bf16x2(ra, rb);
                        }
                        tc::st16(sx + 16 * g, pk);
                    }
                }
                float l0, l1, l2, l3;
                f2_unpack(ls2[0], l0, l1);
                f2_unpack(ls2[1], l2, l3);
                l = l * (resc ? alpha : 1.f) + ((l0 + l1) + (l2 + l3));
            }
            // V(jj) must have landed before this tile's P.V is issued.  Value
            // rows of keys outside [kv_lo, kv_hi) or of blocks not loaded hold
            // stale slots (possibly NaN): each warpgroup zeroes them before its
            // own P.V reads them (both write the same zeros, so whichever
            // product runs first reads zeros)
            const bool landed = mbar_wait(&v_full[ks], (T / kStages) & 1, p.wait_ns);
            if (__any_sync(0xffffffffu, !landed)) {
                if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                abort = true;
                break;
            }
            // (FP8: the V producer wrote those columns as zeros)
            const bool edge = !kF8 && (mask != (1u << kBlocks) - 1u || tbase < kv_lo ||
                                       tbase + kKeys > kv_hi);
            if (edge) {
                // thread row r < 64 zeroes key row r's first 64 dims, r >= 64
                // the second 64 dims of key row r - 64
                const int kr = row & (kKeys - 1), half = row >> 6;
                const int32_t kp = tbase + kr;
                if (!(kp >= kv_lo && kp < kv_hi && ((mask >> (kr >> 4)) & 1u))) {
                    uint8_t *vs = v_s + ks * kTileBytes + half * kKVRegion + kr * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(vs + c * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x * 2 + buf]);
        }
        if (abort) break;
        const PrefillRowInfo &w = ss->sg.w;
        // epilogue: O / l once the segment's last P.V product is in.  Phases
        // up to its last tile - 3 are known complete here (S of its last tile
        // was issued after P.V of the tile two before), and those of earlier
        // segments too, so wait for the last tile - 1 first: a parity names
        // one phase only when the one before it has completed
        {
            const int32_t Tl = T0 + ntile - 1;
            bool done = ntile < 2 || mbar_wait(&pv_done[x], (Tl - 1) & 1, p.wait_ns);
            done = done && mbar_wait(&pv_done[x], Tl & 1, p.wait_ns);
            if (__any_sync(0xffffffffu, !done)) {
                if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                break;
            } else if (p.sk_ctas > 0 && !ss->sg.whole) {
                // a piece of an item cut by this CTA's run: a partial in the
                // CTA's slot (first or last segment), merged afterwards
                tc::fence_after();
                const size_t pr = (static_cast<size_t>(blockIdx.x) * 2 + ss->sg.slot) * (kQTiles * kRows) +
                                  x * kRows + row;
                float4 *dst = reinterpret_cast<float4 *>(p.sk_o + pr * kD);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r32[32];
                    tc::ld32(ox + c * 32, r32);
                    tc::wait_ld();
                    if (valid_row) {
                        const float vs = kF8 ? p.v_scale : 1.f;
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[c * 8 + v] = make_float4(__uint_as_float(r32[4 * v]) * vs, __uint_as_float(r32[4 * v + 1]) * vs,
                                                         __uint_as_float(r32[4 * v + 2]) * vs, __uint_as_float(r32[4 * v + 3]) * vs);
                    }
                }
                if (valid_row) *reinterpret_cast<float2 *>(p.sk_ml + pr * 2) = make_float2(m_ref, l);
                // the item's pieces: CTAs cf .. cl; per (query tile, warp) the
                // warp whose piece completes last merges their 32 rows (no
                // waiting: the others published theirs before counting)
                __syncwarp();
                const int32_t u = ss->sg.item;
                const int32_t lo = __ldg(p.sk_prefix + u), hi = __ldg(p.sk_prefix + u + 1);
                const int32_t cf = sk_cta_of(p, lo), cl = sk_cta_of(p, hi - 1);
                int last = 0;
                if (lane == 0) {
                    __threadfence();
                    const int old = atomicAdd(p.sk_count + (cf * 2 + x) * 4 + (warp & 3), 1);
                    last = old == cl - cf;
                    if (last) __threadfence();
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last && valid_row) {
                    auto piece = [&](int32_t c) {  // slot 1: the item is not c's first segment
                        const int32_t slot = (c == cf && sk_run_start(p, c) < lo) ? 1 : 0;
                        return (static_cast<size_t>(c) * 2 + slot) * (kQTiles * kRows) + x * kRows + row;
                    };
                    float M = -INFINITY, lsum = 0.f;
                    for (int32_t c = cf; c <= cl; ++c) M = fmaxf(M, __ldcg(p.sk_ml + piece(c) * 2));
                    if (M != -INFINITY)
                        for (int32_t c = cf; c <= cl; ++c) {
                            const size_t pc = piece(c);
                            const float mc = __ldcg(p.sk_ml + pc * 2);
                            if (mc != -INFINITY) lsum = fmaf(fast_exp2(mc - M), __ldcg(p.sk_ml + pc * 2 + 1), lsum);
                        }
                    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out) +
                                 ((static_cast<int64_t>(__ldg(p.cu_q_lens + w.r)) + w.i0 + t) * p.hq +
                                  w.g * G + row % G) * (kD / 8);
                    // 32 dims at a time
#pragma unroll 1
                    for (int d0 = 0; d0 < kD; d0 += 32) {
                        float acc[32];
#pragma unroll
                        for (int d = 0; d < 32; ++d) acc[d] = 0.f;
                        if (M != -INFINITY)
                            for (int32_t c = cf; c <= cl; ++c) {
                                const size_t pc = piece(c);
                                const float mc = __ldcg(p.sk_ml + pc * 2);
                                if (mc == -INFINITY) continue;
                                const float wgt = fast_exp2(mc - M);
                                const float4 *src = reinterpret_cast<const float4 *>(p.sk_o + pc * kD + d0);
#pragma unroll
                                for (int v = 0; v < 8; ++v) {
                                    const float4 o4 = __ldcg(src + v);
                                    acc[4 * v] = fmaf(wgt, o4.x, acc[4 * v]);
                                    acc[4 * v + 1] = fmaf(wgt, o4.y, acc[4 * v + 1]);
                                    acc[4 * v + 2] = fmaf(wgt, o4.z, acc[4 * v + 2]);
                                    acc[4 * v + 3] = fmaf(wgt, o4.w, acc[4 * v + 3]);
                                }
                            }
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 o;
                            o.x = pack_bf16x2(acc[8 * v + 0] * inv, acc[8 * v + 1] * inv);
                            o.y = pack_bf16x2(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv);
                            o.z = pack_bf16x2(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv);
                            o.w = pack_bf16x2(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv);
                            dst[d0 / 8 + v] = o;
                        }
                    }
                }
            } else if (split) {
                // a partial: O unnormalised with its reference max and sum
                tc::fence_after();
                const size_t pi = ((static_cast<size_t>(w.r) * p.max_q_len + w.i0 + t) * p.hq +
                                   w.g * G + row % G) * p.kv_splits + w.s;
                float4 *dst = reinterpret_cast<float4 *>(p.ws_o + pi * kD);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r32[32];
                    tc::ld32(ox + c * 32, r32);
                    tc::wait_ld();
                    if (valid_row) {
                        const float vs = kF8 ? p.v_scale : 1.f;
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[c * 8 + v] = make_float4(__uint_as_float(r32[4 * v]) * vs, __uint_as_float(r32[4 * v + 1]) * vs,
                                                         __uint_as_float(r32[4 * v + 2]) * vs, __uint_as_float(r32[4 * v + 3]) * vs);
                    }
                }
                if (valid_row) *reinterpret_cast<float2 *>(p.ws_ml + pi * 2) = make_float2(m_ref, l);
            } else {
                tc::fence_after();
                const float inv = (l > 0.f ? 1.f / l : 0.f) * (kF8 ? p.v_scale : 1.f);
                const int h = row % G;
                uint4 *dst = reinterpret_cast<uint4 *>(p.out) +
                             ((static_cast<int64_t>(__ldg(p.cu_q_lens + w.r)) + w.i0 + t) * p.hq +
                              w.g * G + h) * (kD / 8);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r32[32];
                    tc::ld32(ox + c * 32, r32);
                    tc::wait_ld();
                    if (valid_row) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(r32[8 * v + 0]) * inv, __uint_as_float(r32[8 * v + 1]) * inv);
                            o.y = pack_bf16x2(__uint_as_float(r32[8 * v + 2]) * inv, __uint_as_float(r32[8 * v + 3]) * inv);
                            o.z = pack_bf16x2(__uint_as_float(r32[8 * v + 4]) * inv, __uint_as_float(r32[8 * v + 5]) * inv);
                            o.w = pack_bf16x2(__uint_as_float(r32[8 * v + 6]) * inv, __uint_as_float(r32[8 * v + 7]) * inv);
                            dst[c * 4 + v] = o;
                        }
                    }
                }
            }
        }
        // the next segment: its query tile replaces this one once every
        // product that read it has completed (the waits above)
        tc::fence_before();
        T0 += ntile;
        bool more = false;
        if (lane == 0) {
            SegWalk sw = ss->sw;
            Seg sg;
            more = seg_next(p, qpc, sw, sg);
            if (more) {
                ss->sw = sw;
                ss->sg = sg;
            }
        }
        more = __shfl_sync(0xffffffffu, more, 0);
        __syncwarp();
        if (!more) break;
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// f32, CUDA cores: 16 (query, head) pairs per CTA
// ---------------------------------------------------------------------------
constexpr int kPf32Threads = 128;
constexpr int kPf32Pairs = 16;

__global__ void __launch_bounds__(kPf32Threads) prefill_f32_kernel(const PrefillParams p)
{
    constexpr int NQ = kPf32Pairs;
    extern __shared__ float fsm[];
    const int D = p.head_dim, bs = p.block_size, G = p.group;
    const int qpt = NQ / G;
    float *qs = fsm, *os = qs + NQ * D, *ks = os + NQ * D, *vs = ks + bs * D, *sc = vs + bs * D;
    float *mrow = sc + NQ * bs, *lrow = mrow + NQ, *alpha = lrow + NQ;
    int32_t *phi = reinterpret_cast<int32_t *>(alpha + NQ), *plo = phi + NQ;
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    PrefillRowInfo w;
    if (!prefill_item(p, blockIdx.x, qpt, w)) return;
    const int32_t row0 = __ldg(p.cu_q_lens + w.r) + w.i0;
    if (tid < NQ) {
        const int t = tid / G;
        const bool valid = tid < qpt * G && t < w.nq;
        const int32_t qpos = w.L - w.C + w.i0 + t;
        phi[tid] = valid ? qpos + 1 : 0;
        plo[tid] = p.window > 0 ? max(0, qpos - p.window + 1) : 0;
        mrow[tid] = -INFINITY;
        lrow[tid] = 0.f;
    }
    const float *qg = static_cast<const float *>(p.q);
    for (int i = tid; i < NQ * D; i += kPf32Threads) {
        const int k = i / D, d = i % D, t = k / G, h = k % G;
        const bool valid = k < qpt * G && t < w.nq;
        qs[i] = valid ? qg[(static_cast<int64_t>(row0 + t) * p.hq + w.g * G + h) * D + d] : 0.f;
        os[i] = 0.f;
    }
    __syncthreads();
    const float *kpool = static_cast<const float *>(p.k_pool);
    const float *vpool = static_cast<const float *>(p.v_pool);
    const int32_t *trow = p.tables + static_cast<int64_t>(w.r) * p.width;
    for (int32_t b = w.kv_lo / bs; b * bs < w.kv_hi; ++b) {
        const int32_t blk = b < p.width ? __ldg(trow + b) : -1;
        const bool ok = static_cast<uint32_t>(blk) < static_cast<uint32_t>(p.num_blocks);
        if (!ok && tid == 0) report(p.status, PKV_DEV_BAD_BLOCK);
        if (ok) {
            const int64_t base = (static_cast<int64_t>(blk) * p.hkv + w.g) * bs * D;
            for (int j = tid; j < bs * D; j += kPf32Threads) {
                ks[j] = __ldg(kpool + base + j);
                vs[j] = __ldg(vpool + base + j);
            }
        }
        __syncthreads();
        for (int j = tid; j < NQ * bs; j += kPf32Threads) {
            const int k = j / bs, tt = j % bs;
            const int pos = b * bs + tt;
            float sv = -INFINITY;
            if (ok && pos >= plo[k] && pos < phi[k]) {
                float acc = 0.f;
                for (int d = 0; d < D; ++d) acc = fmaf(qs[k * D + d], ks[tt * D + d], acc);
                sv = acc * p.scale_log2;
            }
            sc[j] = sv;
        }
        __syncthreads();
        if (tid < NQ) {
            float mx = -INFINITY;
            for (int tt = 0; tt < bs; ++tt) mx = fmaxf(mx, sc[tid * bs + tt]);
            const float mn = fmaxf(mrow[tid], mx);
            const float mu = mn == -INFINITY ? 0.f : mn;
            const float al = fast_exp2(mrow[tid] - mu);
            float sum = 0.f;
            for (int tt = 0; tt < bs; ++tt) {
                const float e = fast_exp2(sc[tid * bs + tt] - mu);
                sc[tid * bs + tt] = e;
                sum += e;
            }
            lrow[tid] = lrow[tid] * al + sum;
            mrow[tid] = mn;
            alpha[tid] = al;
        }
        __syncthreads();
        for (int j = tid; j < NQ * D; j += kPf32Threads) {
            const int k = j / D, d = j % D;
            float acc = os[j] * alpha[k];
            for (int tt = 0; tt < bs; ++tt) {
                const float wv = sc[k * bs + tt];
                if (wv != 0.f) acc = fmaf(wv, vs[tt * D + d], acc);  // masked slots may hold NaN
            }
            os[j] = acc;
        }
        __syncthreads();
    }
    float *og = static_cast<float *>(p.out);
    for (int j = tid; j < NQ * D; j += kPf32Threads) {
        const int k = j / D, d = j % D, t = k / G, h = k % G;
        if (k >= qpt * G || t >= w.nq) continue;
        const float l = lrow[k];
        og[(static_cast<int64_t>(row0 + t) * p.hq + w.g * G + h) * D + d] = l > 0.f ? os[j] / l : 0.f;
    }
}

// ---------------------------------------------------------------------------
// merge of the key-range runs (bf16, short chunks): one warp per (row, query
// of the chunk, q head).  M = max of the runs' reference maxima; each run is
// weighted by 2^(m_s - M); out = sum w_s O_s / sum w_s l_s.
// ---------------------------------------------------------------------------
constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) prefill_merge_kernel(const PrefillParams p)
{
    constexpr int D = pf::kD;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
    const int64_t total = static_cast<int64_t>(p.batch) * p.max_q_len * p.hq;
    if (item >= total) return;
    const int32_t h = static_cast<int32_t>(item % p.hq);
    const int64_t ri = item / p.hq;
    const int32_t i = static_cast<int32_t>(ri % p.max_q_len);
    const int32_t r = static_cast<int32_t>(ri / p.max_q_len);
    // the chunk length as the prefill kernel clamps it (call inputs: final
    // before the wait, as the prefill kernel waited on earlier work itself)
    const int32_t c0 = __ldg(p.cu_q_lens + r), c1 = __ldg(p.cu_q_lens + r + 1);
    int32_t C = c1 - c0;
    int32_t L = __ldg(p.seq_lens + r);
    L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);
    if (c0 < 0 || C < 0 || C > p.max_q_len || C > L)
        C = c0 < 0 || C < 0 ? 0 : min(min(C, p.max_q_len), L);
    if (i >= C) return;
    pdl_wait();  // the partials come from the prefill kernel just before
    const size_t base = ((static_cast<size_t>(r) * p.max_q_len + i) * p.hq + h) * p.kv_splits;
    float M = -INFINITY;
    for (int32_t s = 0; s < p.kv_splits; ++s) M = fmaxf(M, p.ws_ml[(base + s) * 2]);
    float acc[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    if (M != -INFINITY) {
        for (int32_t s = 0; s < p.kv_splits; ++s) {
            const float2 ml = *reinterpret_cast<const float2 *>(p.ws_ml + (base + s) * 2);
            if (ml.x == -INFINITY) continue;  // an empty run wrote no values
            const float wgt = fast_exp2(ml.x - M);
            lsum = fmaf(wgt, ml.y, lsum);
            const float *src = p.ws_o + (base + s) * D + lane;
#pragma unroll
            for (int e = 0; e < D / 32; ++e) acc[e] = fmaf(wgt, src[32 * e], acc[e]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) +
                         (static_cast<size_t>(c0 + i) * p.hq + h) * D + lane;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) out[32 * e] = __float2bfloat16_rn(acc[e] * inv);
}

// ---------------------------------------------------------------------------
// persistent balanced schedule: the plan (tile prefix sums of the items; the
// cut items' arrival counters zeroed)
// ---------------------------------------------------------------------------
constexpr int kSkPlanThreads = 1024;

__global__ void __launch_bounds__(kSkPlanThreads) prefill_sk_plan_kernel(const PrefillParams p)
{
    __shared__ int32_t warp_sum[kSkPlanThreads / 32];
    __shared__ int32_t carry;
    pdl_wait();  // lengths may come from the previous kernel on the stream
    pdl_trigger();
    const int qpc = pf::kQTiles * (pf::kRows / p.group);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        p.sk_prefix[0] = 0;
    }
    for (int32_t i = threadIdx.x; i < p.sk_ctas * 8; i += kSkPlanThreads) p.sk_count[i] = 0;
    __syncthreads();
    for (int32_t base = 0; base < p.sk_items; base += kSkPlanThreads) {
        const int32_t u = base + threadIdx.x;
        int32_t n = 0;
        PrefillRowInfo w;
        if (u < p.sk_items && prefill_item(p, u, qpc, w))
            n = (w.kv_hi - 1) / pf::kKeys - w.kv_lo / pf::kKeys + 1;
        // inclusive scan: within the warp, then over the warps' sums
        int32_t v = n;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, v, d);
            if (lane >= d) v += o;
        }
        if (lane == 31) warp_sum[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int32_t ws = warp_sum[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t o = __shfl_up_sync(0xffffffffu, ws, d);
                if (lane >= d) ws += o;
            }
            warp_sum[lane] = ws;  // inclusive over the warps
        }
        __syncthreads();
        const int32_t incl = v + (warp > 0 ? warp_sum[warp - 1] : 0) + carry;
        if (u < p.sk_items) p.sk_prefix[u + 1] = incl;
        __syncthreads();
        if (threadIdx.x == kSkPlanThreads - 1) carry = incl;
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool prefill_shape_built(pkv_dtype dtype, int32_t D, int32_t bs, int32_t G)
{
    if (G < 1 || G > 16) return false;
    if (dtype == PKV_BF16 || dtype == PKV_FP8_E4M3) return D == pf::kD && bs == 16 && (pf::kRows % G) == 0;
    return (D == 32 || D == 64 || D == 128 || D == 256) && bs <= 64 && bs * D <= 4096 &&
           (kPf32Pairs % G) == 0;
}

int32_t prefill_queries_per_cta(pkv_dtype dtype, int32_t G)
{
    return dtype != PKV_F32 ? pf::kQTiles * (pf::kRows / G) : kPf32Pairs / G;
}

PrefillSplit prefill_split_plan(int32_t batch, int32_t hq, int32_t hkv, int32_t D, int32_t bs,
                                int32_t max_q_len, int32_t max_seq_len, int32_t window, int num_sms)
{
    PrefillSplit sp{1, 0};
    if (hkv <= 0 || hq % hkv != 0 || batch <= 0 || max_q_len <= 0) return sp;
    const int32_t G = hq / hkv;
    if (D != pf::kD || bs != 16 || G < 1 || pf::kRows % G != 0) return sp;
    if (max_q_len > pf::kRows / G) return sp;  // chunks that need both query tiles: no split
    const int64_t ctas = static_cast<int64_t>(batch) * hkv;
    const int64_t keys = window > 0 ? std::min<int64_t>(max_seq_len, static_cast<int64_t>(window) + max_q_len)
                                    : max_seq_len;
    // +1: a CTA's range may start inside a tile
    const int64_t tiles = (keys + pf::kKeys - 1) / pf::kKeys + 1;
    // about four CTAs per SM over the grid, at least 8 tiles (512 keys) per run
    int64_t s = (4ll * std::max(num_sms, 1) + ctas - 1) / ctas;
    s = std::min<int64_t>(s, tiles / 8);
    s = std::max<int64_t>(1, std::min<int64_t>(s, 32));
    if (s == 1) return sp;
    sp.splits = static_cast<int32_t>(s);
    sp.tiles = static_cast<int32_t>((tiles + s - 1) / s);
    return sp;
}

int32_t prefill_sk_ctas(pkv_dtype dtype, int32_t batch, int32_t hq, int32_t hkv, int32_t D, int32_t bs,
                        int32_t max_q_len, int num_sms)
{
    if (dtype == PKV_F32 || hkv <= 0 || hq % hkv != 0 || batch <= 0 || max_q_len <= 0 || num_sms <= 0)
        return 0;
    const int32_t G = hq / hkv;
    if (D != pf::kD || bs != 16 || G < 1 || pf::kRows % G != 0) return 0;
    if (max_q_len <= pf::kRows / G) return 0;  // one query tile: the key-range runs serve it
    const int64_t qpc = static_cast<int64_t>(pf::kQTiles) * (pf::kRows / G);
    const int64_t items = static_cast<int64_t>(batch) * hkv * ((max_q_len + qpc - 1) / qpc);
    // more items than SMs (else one wave of one CTA per item already fits),
    // and a plan the one-CTA plan kernel scans quickly
    if (items <= num_sms || items > 65536) return 0;
    return num_sms;
}

size_t prefill_sk_ws_bytes(int32_t items, int32_t ctas)
{
    if (ctas <= 0) return 0;
    const size_t pre = ((static_cast<size_t>(items + 1) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255)) +
                       ((static_cast<size_t>(ctas) * 8 * sizeof(int32_t) + 255) & ~static_cast<size_t>(255));
    const size_t rows = static_cast<size_t>(ctas) * 2 * pf::kQTiles * pf::kRows;
    const size_t o = (rows * pf::kD * sizeof(float) + 255) & ~static_cast<size_t>(255);
    return pre + o + rows * 2 * sizeof(float);
}

size_t prefill_split_ws_bytes(int32_t batch, int32_t hq, int32_t max_q_len, const PrefillSplit &sp)
{
    if (sp.splits <= 1) return 0;
    const size_t n = static_cast<size_t>(batch) * max_q_len * hq * sp.splits;
    const size_t o = (n * pf::kD * sizeof(float) + 255) & ~static_cast<size_t>(255);
    return o + n * 2 * sizeof(float);
}

template <bool kF8>
static cudaError_t launch_prefill_tc(const PrefillParams &p, const CUtensorMap &kmap,
                                    const CUtensorMap &vmap, cudaStream_t stream)
{
    const int64_t ctas = p.sk_ctas > 0 ? p.sk_ctas
                                       : static_cast<int64_t>(p.batch) * p.hkv * p.q_tiles * p.kv_splits;
    if (ctas == 0) return cudaSuccess;
    constexpr int smem = pf::Layout<kF8>::kLaunchBytes;
    cudaError_t err = cudaFuncSetAttribute(prefill_kernel<kF8>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_PREFILL, stream);
    if (p.sk_ctas > 0)
        err = launch_pdl(prefill_sk_plan_kernel, dim3(1), dim3(kSkPlanThreads), 0, stream, p);
    if (err == cudaSuccess)
        err = launch_pdl(prefill_kernel<kF8>, dim3(static_cast<unsigned>(ctas)), dim3(pf::kThreads), smem,
                         stream, kmap, vmap, p);
    if (err == cudaSuccess && p.kv_splits > 1) {
        const int64_t items = static_cast<int64_t>(p.batch) * p.max_q_len * p.hq;
        err = launch_pdl(prefill_merge_kernel,
                         dim3(static_cast<unsigned>((items + kMergeWarps - 1) / kMergeWarps)),
                         dim3(kMergeWarps * 32), 0, stream, p);
    }
    prof_end(PKV_KERNEL_PREFILL, stream);
    return err;
}

cudaError_t launch_prefill_bf16(const PrefillParams &p, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, cudaStream_t stream)
{
    return launch_prefill_tc<false>(p, kmap, vmap, stream);
}

cudaError_t launch_prefill_fp8(const PrefillParams &p, cudaStream_t stream)
{
    const CUtensorMap none{};  // the FP8 producers read the pools by bulk copy
    return launch_prefill_tc<true>(p, none, none, stream);
}

cudaError_t launch_prefill_f32(const PrefillParams &p, cudaStream_t stream)
{
    const int64_t ctas = static_cast<int64_t>(p.batch) * p.hkv * p.q_tiles;
    if (ctas == 0) return cudaSuccess;
    const int D = p.head_dim, bs = p.block_size, NQ = kPf32Pairs;
    const size_t smem = sizeof(float) * (2 * NQ * D + 2 * bs * D + NQ * bs + 3 * NQ) +
                        sizeof(int32_t) * 2 * NQ;
    cudaError_t err = cudaFuncSetAttribute(prefill_f32_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_PREFILL, stream);
    err = launch_pdl(prefill_f32_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kPf32Threads),
                     smem, stream, p);
    prof_end(PKV_KERNEL_PREFILL, stream);
    return err;
}

}  // namespace pkv
