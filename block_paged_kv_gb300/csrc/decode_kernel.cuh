// Split-KV paged decode attention for bf16 and FP8 pools ("perf.md": the paged decode
// reads the pages through the block table and splits each row into partitions
// whose online-softmax partials a reducer merges; all q heads of a GQA group
// share each block load, as the pages' grouped decode kernels do).
//
// One launch carries two kinds of CTA, one work item each:
//   prefix item (the first n_prefix_ctas CTAs): group, kv head g, row chunk,
//       prefix split s -> prefix blocks s*Cp ..; its four query tiles hold
//       (row, head) pairs of the group's rows, so every shared block is read
//       once for all of them;
//   split item: row r, kv head g, split s -> blocks b_first + s*C .. ; its one
//       query tile holds the G q heads of (r, g) (a verify step: the G heads
//       of each of the row's few queries).
// K and V (block, kv head) tiles are brought into shared memory with one TMA
// tensor load each (5-D maps viewing [block][kv head][slot][dim] as
// (64 dims, slot, 64-dim region, kv head, block), 128-byte swizzle, so a tile
// lands as one 2 KiB swizzled region per 64 dims) that completes on an mbarrier.
//   split item: each of the four warps takes every fourth block of the run and
//       keeps its own ring of stages: it issues the loads of its next blocks
//       itself as it frees a stage, so no warp ever waits behind another;
//   prefix item: the four warps share one ring (each owns a query tile and
//       reads every block); warp 0 refills a stage once all four released it.
// Warps compute the transposed products S^T = K Q^T and O^T = V^T P^T with
// mma.sync m16n8k16 (fp32 accumulate), so that a block's 16 tokens (S^T) and
// 16-dim slices of the head (O^T) fill the 16-row M side and the query rows
// (the G q heads of a GQA group, G <= 8 in one n-tile of 8, or two n-tiles)
// sit on N: a decode step of G <= 8 heads wastes no M rows, and the query's
// fragments are small enough to stay in registers.  The online softmax runs
// on the accumulator fragments, a column per query row, with shuffles across
// the 8 lanes that share it.  Each tile's partial (max in log2 units, sum,
// unnormalised O) goes to the workspace.
//   bf16 pools: K rows and V^T columns come out of the swizzled tiles with
//       ldmatrix (plain for K, transposing for V); P enters the P.V product
//       as two bf16 terms (hi + lo) so that its rounding stays far below the
//       output's own bf16 rounding.
//   FP8 pools ("perf.md", quantisation scheme table: FP8 KV cache with
//       per-layer scales): a (block, kv head) tile is one contiguous run of
//       16 * D bytes, brought in with one bulk copy; its bytes are already in
//       fragment order, so each lane reads its operands as 16-byte words and
//       widens them to f16 (exact) in registers.  The query is converted to
//       f16 once, P enters P.V as one f16 term (2^-11 relative), the K scale
//       is folded into the score scale and the V scale applied to the partial.
#pragma once

#include "decode_common.cuh"

namespace pkv {

template <int D, bool kF8, int NQ>
struct KvCfg {
    static constexpr int kTok = 16;                       // block_size
    static constexpr int kElem = kF8 ? 1 : 2;             // bytes per K/V element
    static constexpr int kTileBytes = kTok * D * kElem;   // one (block, kv head) tile of K or V
    // blocks per pipeline stage: an FP8 stage at head_dim <= 128 holds two
    // blocks, so that each pass of the online softmax covers 32 tokens and
    // the per-pass costs (waits, reductions, rescale, refill) are paid once
    // per 32 tokens
    static constexpr int kBps = (kF8 && D <= 128) ? 2 : 1;
    static constexpr int kStageBytes = kBps * 2 * kTileBytes;  // K + V of each block
    static constexpr int kTR = 8 * NQ;                    // query rows of a warp tile (N side)
    // the query's B fragments stay in registers (D/16 k-steps x NQ n-tiles x
    // 2 words) unless that is 64 words or more; in registers, the query tiles
    // are staged through the ring before the first load, otherwise they keep
    // a region of their own
    static constexpr bool kQInRegs = D * NQ <= 256;
    static constexpr int kTiles = 4;                      // query tiles of a prefix item
    // ring sized so that kCtasPerSm CTAs fit on an SM: three when the query
    // lives in registers (a CTA's start - lengths, tables, query, first loads
    // - then overlaps two others' streaming; measured 6 % faster than two
    // CTAs with a 96 KB ring at head_dim 128), otherwise two (the query tiles
    // need their own region)
    static constexpr int kRingBytes = 64 * 1024;
    static constexpr int kCtasPerSm = kQInRegs ? 3 : 2;
    static constexpr int kStages = kRingBytes / kStageBytes;
    static constexpr int kStagesPerWarp = kStages / kDecodeWarps;  // split items
    static_assert(kStages % kDecodeWarps == 0, "split items give each warp the same stages");
    static constexpr int kRegions = D / 64;               // 64-dim swizzled regions per tile
    static constexpr int kRegionBytes = kTok * 128;
    static constexpr int kQStride = (D + 8) * 2;          // padded query row (bytes)
    static constexpr int kQTileBytes = kTR * kQStride;
    static constexpr int kMT = D / 16;                    // 16-dim m-tiles of O^T
    static constexpr int kKS = D / 16;                    // 16-dim k-steps of K Q^T
};

template <int D, bool kF8, int NQ>
struct KvSmem {
    using C = KvCfg<D, kF8, NQ>;
    static constexpr int kStageOff = 0;
    static constexpr int kQOff = C::kQInRegs ? 0 : C::kRingBytes;
    static constexpr int kBarOff =
        C::kQInRegs ? C::kRingBytes : C::kRingBytes + C::kTiles * C::kQTileBytes;
    static constexpr int kOkOff = kBarOff + 2 * C::kStages * 8;
    static constexpr int kPairOff = kOkOff + C::kStages * C::kBps * 4;
    static constexpr int kMiscOff = kPairOff + 3 * C::kTiles * C::kTR * 4;
    static constexpr int kBytes = kMiscOff + 16;
    static constexpr int kLaunchBytes = kBytes + 1024;  // room to align the base to 1024
    static_assert(C::kTiles * C::kQTileBytes <= C::kRingBytes || !C::kQInRegs,
                  "query tiles staged through the ring fit in it");
    static_assert(kDecodeWarps * C::kTR * D * 4 + kDecodeWarps * C::kTR * 8 <= kBarOff,
                  "the merge buffers fit below the barriers");
};

// Swizzled shared address of the 16-byte chunk holding dims d0..d0+7 of token
// `tok` in a K/V tile (TMA SWIZZLE_128B: chunk index XOR (line % 8)).
__device__ __forceinline__ uint32_t kv_chunk_addr(uint32_t tile, int tok, int d0)
{
    return tile + (d0 >> 6) * (16 * 128) + tok * 128 +
           ((((d0 & 63) >> 3) ^ (tok & 7)) << 4);
}

// Block ids of a strided run, fetched 32 at a time ahead of use: index j of
// the run is row[first + stride * j].  All lanes call next() with the same,
// increasing j; the id comes back on every lane.
struct BlockIds {
    const int32_t *row;
    int32_t first, stride, n, batch_no;
    int32_t cur, nxt;
    __device__ __forceinline__ int32_t fetch(int32_t j, int lane) const
    {
        const int32_t k = j + lane;
        return k < n ? __ldg(row + first + stride * k) : -1;
    }
    __device__ __forceinline__ void init(const int32_t *r, int32_t f, int32_t s, int32_t count,
                                         int lane)
    {
        row = r;
        first = f;
        stride = s;
        n = count;
        batch_no = 0;
        cur = fetch(0, lane);
        nxt = fetch(32, lane);
    }
    __device__ __forceinline__ int32_t next(int32_t j, int lane)
    {
        if ((j >> 5) != batch_no) {
            cur = nxt;
            ++batch_no;
            nxt = fetch((batch_no + 1) * 32, lane);
        }
        return __shfl_sync(0xffffffffu, cur, j & 31);
    }
};

// The work of CTA `cta` of one decode call (p), its K/V tensor maps (bf16)
// given by reference to kernel-parameter memory.
template <int D, bool kMQ, bool kF8, int NQ>
__device__ __forceinline__ void decode_split_body(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                                  const DecodeParams &p, const int64_t cta)
{
    using C = KvCfg<D, kF8, NQ>;
    using SM = KvSmem<D, kF8, NQ>;
    constexpr int NW = kDecodeWarps;
    constexpr int STAGES = C::kStages;
    constexpr int SPW = C::kStagesPerWarp;
    constexpr int TR = C::kTR;  // query rows per warp tile: the N side, NQ n-tiles of 8

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stage_mem = smem + SM::kStageOff;
    uint8_t *q_mem = smem + SM::kQOff;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::kBarOff);
    uint64_t *empty = full + STAGES;
    int32_t *stage_ok = reinterpret_cast<int32_t *>(smem + SM::kOkOff);
    int32_t *pair_row = reinterpret_cast<int32_t *>(smem + SM::kPairOff);
    int32_t *pair_head = pair_row + C::kTiles * TR;
    int32_t *pair_len = pair_head + C::kTiles * TR;
    int32_t *misc = reinterpret_cast<int32_t *>(smem + SM::kMiscOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int bs = C::kTok;

    if (!kF8 && threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    pdl_wait();     // inputs may come from the previous kernel on the stream
    pdl_trigger();  // the merge kernel may be scheduled now; it waits for us

    // ---------------------------------------------------------------- work item
    const bool prefix_item = cta < p.plan.n_prefix_ctas;
    int32_t b0, nblk, slot, tab_row, g, lo_all, hi_all, tiles;
    // split item only: the row, its query count and first packed query
    int32_t row_r = 0, row_C = 1, row_q0 = 0;
    // query rows of a split item: the G heads of one query (decode), or
    // (query, head) pairs of a row's few queries (kMQ: a verify step); the
    // launch takes NQ so that R <= TR
    const int R = kMQ ? G * p.max_q : G;
    // the block ids of the run (this warp's share of a split item; the whole
    // run for a prefix item, fetched by warp 0)
    BlockIds ids;
    // B fragments of Q^T (query rows on N, NQ n-tiles of 8):
    // b0 = Q[row 8n + lane/4][16kk + 2(lane%4), +1], b1 = the same 8 dims further.
    // A split item whose query fits in registers loads them straight from
    // global memory (no shared-memory staging, no wait before its first
    // block loads); other items stage the query tiles in shared memory.
    uint32_t qb[C::kQInRegs ? C::kKS : 1][NQ][2];
    const bool q_direct = C::kQInRegs && !prefix_item;
    auto load_q_direct = [&]() {
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
            const int row = 8 * n + (lane >> 2);
            int32_t qr = -1, qh = 0;
            if constexpr (kMQ) {
                if (row < R && row / G < row_C) {
                    qr = row_q0 + row / G;
                    qh = g * G + row % G;
                }
            } else if (row < G) {
                qr = row_r;
                qh = g * G + row;
            }
            const uint32_t *src = reinterpret_cast<const uint32_t *>(p.q) +
                                  (static_cast<int64_t>(qr < 0 ? 0 : qr) * p.hq + qh) * (D / 2) + (lane & 3);
#pragma unroll
            for (int kk = 0; kk < C::kKS; ++kk) {
                qb[kk][n][0] = qr >= 0 ? __ldg(src + 8 * kk) : 0u;
                qb[kk][n][1] = qr >= 0 ? __ldg(src + 8 * kk + 4) : 0u;
            }
        }
    };
    if (!prefix_item) {
        int64_t bid = cta - p.plan.n_prefix_ctas;
        const int32_t s = static_cast<int32_t>(bid % p.plan.n_suffix_splits);
        bid /= p.plan.n_suffix_splits;
        g = static_cast<int32_t>(bid % p.hkv);
        row_r = static_cast<int32_t>(bid / p.hkv);
        const int32_t *table_row = p.tables + static_cast<int64_t>(row_r) * p.width;
        // This warp's block ids are fetched before the row's length is known,
        // on the guess that the row's own splits start at block 0 (full
        // attention, no shared prefix), so that the two fetches overlap; a
        // decode step's query loads go out with them.
        const int32_t b_guess = s * p.plan.split_blocks;
        const int32_t n_guess =
            max(0, (min(p.plan.split_blocks, p.width - b_guess) - warp + NW - 1) / NW);
        ids.init(table_row + (n_guess > 0 ? b_guess : 0), warp, NW, n_guess, lane);
        if constexpr (C::kQInRegs && !kMQ) load_q_direct();
        const RowRange rr = row_range(p, row_r, s == 0 && g == 0);
        b0 = rr.b_first + s * p.plan.split_blocks;
        const int32_t b1 = min(b0 + p.plan.split_blocks, rr.b_end);
        if (b0 >= b1) return;
        nblk = b1 - b0;
        slot = p.plan.n_prefix_splits + s;
        tab_row = row_r;
        lo_all = rr.lo;
        hi_all = rr.L;
        row_C = rr.C;
        row_q0 = rr.q0;
        tiles = 1;
        if constexpr (C::kQInRegs && kMQ) load_q_direct();
        const int32_t nbw = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;
        if (rr.b_first != 0)
            ids.init(table_row + b0, warp, NW, nbw, lane);  // the guess was wrong
        else
            ids.n = nbw;  // fetched ids past the run are never used
    } else {
        tiles = C::kTiles;
        int64_t bid = cta;
        const int32_t s = static_cast<int32_t>(bid % p.plan.n_prefix_splits);
        bid /= p.plan.n_prefix_splits;
        g = static_cast<int32_t>(bid % p.hkv);
        bid /= p.hkv;
        const int32_t chunk = static_cast<int32_t>(bid % p.plan.prefix_chunks);
        const int32_t grp = static_cast<int32_t>(bid / p.plan.prefix_chunks);
        int32_t P = __ldg(p.prefix_blocks + grp);
        const int32_t pmax = p.plan.prefix_max;
        P = P < 0 ? 0 : (P > pmax ? pmax : P);
        b0 = s * p.plan.prefix_split_blocks;
        const int32_t b1 = min(b0 + p.plan.prefix_split_blocks, P);
        if (b0 >= b1) return;
        nblk = b1 - b0;
        slot = s;
        for (int i = threadIdx.x; i < tiles * TR; i += blockDim.x) pair_row[i] = -1;
        __syncthreads();
        if (warp == 0) {
            // rows of the group in ascending order; pair k = rank * G + j
            const int32_t per_cta = tiles * TR;
            const int32_t kbase = chunk * per_cta;
            int32_t cnt = 0, leader = -1, hmax = 0;
            for (int32_t base = 0; base < p.batch; base += 32) {
                const int32_t r = base + lane;
                const bool in = r < p.batch && __ldg(p.group_of_row + r) == grp;
                const uint32_t m = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const int32_t rank = cnt + __popc(m & ((1u << lane) - 1u));
                    if (rank == 0) leader = r;
                    int32_t L = __ldg(p.seq_lens + r);
                    L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);
                    if (L < P * bs) report(p.status, PKV_DEV_BAD_PREFIX);
                    if ((rank + 1) * G > p.plan.prefix_chunks * per_cta)
                        report(p.status, PKV_DEV_BAD_PREFIX);  // more rows than max_group_rows
                    for (int j = 0; j < G; ++j) {
                        const int32_t k = rank * G + j - kbase;
                        if (k >= 0 && k < per_cta) {
                            pair_row[k] = r;
                            pair_head[k] = g * G + j;
                            pair_len[k] = L;
                            hmax = max(hmax, L);
                        }
                    }
                }
                cnt += __popc(m);
            }
            leader = __reduce_max_sync(0xffffffffu, leader);
            hmax = __reduce_max_sync(0xffffffffu, hmax);
            if (lane == 0) {
                misc[0] = leader;
                misc[1] = hmax;
            }
        }
        __syncthreads();
        if (pair_row[0] < 0) return;  // this chunk lies past the group's rows
        tab_row = misc[0];
        lo_all = 0;
        hi_all = misc[1];
        // every row of the chunk must hold the leader's blocks in this range
        for (int i = threadIdx.x; i < tiles * TR * nblk; i += blockDim.x) {
            const int k = i / nblk, b = b0 + i % nblk;
            const int32_t pr = pair_row[k];
            if (pr >= 0 && (k % G) == 0 &&
                __ldg(p.tables + static_cast<int64_t>(pr) * p.width + b) !=
                    __ldg(p.tables + static_cast<int64_t>(tab_row) * p.width + b))
                report(p.status, PKV_DEV_BAD_PREFIX);
        }
    }

    // ------------------------------------------------- query tiles + barriers
    {
        constexpr int kVec = D / 8;  // 16-byte vectors per row
        const int qrows = q_direct ? 0 : (prefix_item ? tiles * TR : TR);
        for (int i = threadIdx.x; i < qrows * kVec; i += blockDim.x) {
            const int row = i / kVec, v = i % kVec;
            int32_t qr = -1, qh = 0;
            if (!prefix_item) {
                if constexpr (kMQ) {
                    if (row < R && row / G < row_C) {
                        qr = row_q0 + row / G;
                        qh = g * G + row % G;
                    }
                } else if (row < G) {
                    qr = row_r;
                    qh = g * G + row;
                }
            } else {
                qr = pair_row[row];
                qh = pair_head[row];
            }
            uint4 val = make_uint4(0, 0, 0, 0);
            if (qr >= 0)
                val = __ldg(reinterpret_cast<const uint4 *>(p.q) +
                            ((static_cast<int64_t>(qr) * p.hq + qh) * D) / 8 + v);
            if constexpr (kF8) {
                // bf16 -> f16 (exact inside the f16 range; NaN stays NaN)
                uint32_t w[4] = {val.x, val.y, val.z, val.w};
                bool bad = false;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = bf16lo_to_f32(w[i]), hi = bf16hi_to_f32(w[i]);
                    bad |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
                    w[i] = pack_f16x2(lo, hi);
                }
                if (bad) report(p.status, PKV_DEV_Q_RANGE);
                val = make_uint4(w[0], w[1], w[2], w[3]);
            }
            const int qt = prefix_item ? row / TR : 0, qr_in = prefix_item ? row % TR : row;
            *reinterpret_cast<uint4 *>(q_mem + qt * C::kQTileBytes + qr_in * C::kQStride + v * 16) =
                val;
        }
        if (threadIdx.x == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], NW);  // prefix items: every warp releases every stage
            }
            fence_mbar_init();
        }
        __syncthreads();
    }

    // a split item's warps all read query tile 0; a prefix item's warp w owns
    // tile w
    const int tile = prefix_item ? warp : 0;
    const uint32_t qb_lane = smem_u32(q_mem + tile * C::kQTileBytes) + (lane >> 2) * C::kQStride +
                             (lane & 3) * 4;
    if constexpr (C::kQInRegs) {
        if (!q_direct) {
            // a prefix item's tiles, staged through the ring
#pragma unroll
            for (int kk = 0; kk < C::kKS; ++kk)
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    const uint32_t a = qb_lane + n * 8 * C::kQStride + kk * 32;
                    qb[kk][n][0] = lds32(a);
                    qb[kk][n][1] = lds32(a + 16);
                }
            // the ring is about to be overwritten by TMA (async proxy) after
            // these generic-proxy reads and writes of the staged query tiles
            fence_proxy_async_smem();
            __syncthreads();
        }
    }

    // ------------------------------------------------------------- loads
    // A stage holds BPS blocks; pass k of the loop below consumes one stage.
    // split item: warp w's blocks are b0 + w + NW*j (j = 0 .. nb-1); its pass
    //   k covers j = BPS*k .. BPS*k + BPS-1 and goes to stage w*SPW + k % SPW.
    // prefix item: block j of the run, pass k covers j = BPS*k ..; stage
    //   k % STAGES; loads issued by warp 0.
    constexpr int BPS = C::kBps;
    const uint64_t policy = l2_evict_first_policy();
    const int32_t nb = prefix_item ? nblk : (nblk > warp ? (nblk - warp + NW - 1) / NW : 0);
    const int32_t nk = (nb + BPS - 1) / BPS;
    const bool issuer = !prefix_item || warp == 0;
    if (prefix_item && warp == 0)
        ids.init(p.tables + static_cast<int64_t>(tab_row) * p.width + b0, 0, 1, nb, lane);
    auto stage_of = [&](int32_t k) { return prefix_item ? k % STAGES : warp * SPW + k % SPW; };
    // diagnostic drill: pass 0's loads are never issued (its wait runs out)
    auto withheld = [&](int32_t k) { return (p.drill & kDrillWithholdFirst) != 0 && k == 0; };
    auto issue = [&](int32_t k) {  // whole warp; lane 0 issues
        int32_t bj[BPS];
#pragma unroll
        for (int i = 0; i < BPS; ++i) bj[i] = ids.next(k * BPS + i, lane);  // -1 past the run
        if (lane == 0 && !withheld(k)) {
            const int st = stage_of(k);
            bool okv[BPS];
            uint32_t bytes = 0;
#pragma unroll
            for (int i = 0; i < BPS; ++i) {
                const bool exists = k * BPS + i < nb;
                okv[i] = exists && static_cast<uint32_t>(bj[i]) < static_cast<uint32_t>(p.num_blocks);
                if (exists && !okv[i]) report(p.status, PKV_DEV_BAD_BLOCK);
                stage_ok[st * BPS + i] = okv[i] ? 1 : 0;
                bytes += okv[i] ? 2 * C::kTileBytes : 0;
            }
            if (bytes == 0) {
                mbar_arrive(&full[st]);
            } else {
                mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
                for (int i = 0; i < BPS; ++i) {
                    if (!okv[i]) continue;
                    uint8_t *kdst = stage_mem + st * C::kStageBytes + i * 2 * C::kTileBytes;
                    uint8_t *vdst = kdst + C::kTileBytes;
                    if constexpr (kF8) {
                        // the tile is one contiguous run of the pool
                        const int64_t off = (static_cast<int64_t>(bj[i]) * p.hkv + g) * C::kTileBytes;
                        bulk_load(kdst, static_cast<const uint8_t *>(p.k_pool) + off, C::kTileBytes,
                                  &full[st], policy);
                        bulk_load(vdst, static_cast<const uint8_t *>(p.v_pool) + off, C::kTileBytes,
                                  &full[st], policy);
                    } else {
                        // one box per (block, kv head) tile: every 64-dim region at once
                        tma_load_5d(kdst, &kmap, &full[st], 0, 0, 0, g, bj[i], policy);
                        tma_load_5d(vdst, &vmap, &full[st], 0, 0, 0, g, bj[i], policy);
                    }
                }
            }
        }
    };
    const int32_t depth = prefix_item ? STAGES : SPW;
    if (issuer)
        for (int32_t k = 0; k < min(depth, nk); ++k) issue(k);
    // wind-down after a wait ran out: the loads this warp issued and nobody
    // consumed, passes k0 .. k_end-1, land before it leaves (their stages are
    // then quiet when the ring is reused or the CTA exits).  While pass k
    // is awaited, the passes below min(k + depth, nk) have been issued.
    auto drain = [&](int32_t k0, int32_t k_end) {
        if (issuer && lane == 0)
            for (int32_t j = k0; j < min(k_end, nk); ++j)
                if (!withheld(j)) mbar_wait(&full[stage_of(j)], (j / depth) & 1);
        __syncwarp();
    };
    if constexpr (kF8 && C::kQInRegs) {
        if (q_direct) {
            // bf16 -> f16 (exact inside the f16 range; NaN stays NaN), while
            // the first loads are in flight
            bool bad = false;
#pragma unroll
            for (int kk = 0; kk < C::kKS; ++kk)
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    qb[kk][n][0] = bf16x2_to_f16x2(qb[kk][n][0], bad);
                    qb[kk][n][1] = bf16x2_to_f16x2(qb[kk][n][1], bad);
                }
            if (bad) report(p.status, PKV_DEV_Q_RANGE);
        }
    }

    // ---------------------------------------------------------------- compute
    // split item: the four warps' partials of the one tile meet in the ring
    // (free once every warp is past its last block)
    float *mbuf = reinterpret_cast<float *>(stage_mem);  // [NW][R][D]
    float *mlbuf = mbuf + NW * TR * D;                    // [NW][R][2], R <= TR
    const int g8 = lane >> 2;  // A rows g8, g8 + 8; B / C column g8 (B), 2cc (C)
    const int cc = lane & 3;
    // bf16 ldmatrix rows of this lane (matrix lane/8, row lane%8): K as the A
    // operand of S^T (tokens 0-7 / 8-15 at dims +0 / +8: plain), V as that of
    // O^T (the same, transposed on the way: dims +0 / +8 at tokens 0-7 / 8-15)
    const int ka_tok = ((lane >> 3) & 1) * 8 + (lane & 7), ka_dof = (lane >> 4) * 8;
    const int va_tok = (lane >> 4) * 8 + (lane & 7), va_dof = ((lane >> 3) & 1) * 8;
    // key range of this lane's C columns: query rows 8n + 2cc + e
    int clo[NQ][2], chi[NQ][2];
#pragma unroll
    for (int n = 0; n < NQ; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = 8 * n + 2 * cc + e;
            int lo = 0, hi = 0;
            if (prefix_item) {
                const int kq = tile * TR + row;
                hi = pair_row[kq] >= 0 ? pair_len[kq] : 0;
            } else if constexpr (kMQ) {
                const int t = row / G;
                hi = (row < R && t < row_C) ? hi_all - row_C + t + 1 : 0;
                lo = (p.window > 0 && hi > 0) ? max(0, hi - p.window) : 0;
            } else if (row < R) {
                lo = lo_all;
                hi = hi_all;
            }
            clo[n][e] = lo;
            chi[n][e] = hi;
        }
    float oT[C::kMT][NQ][4];  // [16-dim m-tile][n-tile][C fragment]
#pragma unroll
    for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
        for (int n = 0; n < NQ; ++n) oT[mt][n][0] = oT[mt][n][1] = oT[mt][n][2] = oT[mt][n][3] = 0.f;
    float mc[NQ][2], lc[NQ][2];
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
        mc[n][0] = mc[n][1] = -INFINITY;
        lc[n][0] = lc[n][1] = 0.f;
    }

    for (int32_t k = 0; k < nk; ++k) {
        const int st = stage_of(k);
        const int32_t use = prefix_item ? k / STAGES : k / SPW;
        const bool got = mbar_wait(&full[st], use & 1, p.wait_ns);
        if (__any_sync(0xffffffffu, !got)) {
            if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
            drain(k, k + depth);
            break;
        }
        const uint32_t stile = smem_u32(stage_mem + st * C::kStageBytes);
        bool okb[BPS];
        int base_tok[BPS];
#pragma unroll
        for (int i = 0; i < BPS; ++i) {
            okb[i] = stage_ok[st * BPS + i] != 0;
            const int32_t j = k * BPS + i;
            base_tok[i] = (b0 + (prefix_item ? j : warp + NW * j)) * bs;
        }

        // S^T = K Q^T: rows = the block's tokens g8 (first half) and
        // g8 + 8 (second half); even and odd 16-dim steps in two chains
        float sT[BPS][NQ][4];
#pragma unroll
        for (int i = 0; i < BPS; ++i) {
            const uint32_t kt = stile + i * 2 * C::kTileBytes;
            float sa[2][NQ][4] = {};
            auto q_frag = [&](int kk, int n, uint32_t &b0, uint32_t &b1) {
                if constexpr (C::kQInRegs) {
                    b0 = qb[kk][n][0];
                    b1 = qb[kk][n][1];
                } else {
                    const uint32_t qa = qb_lane + n * 8 * C::kQStride + kk * 32;
                    b0 = lds32(qa);
                    b1 = lds32(qa + 16);
                }
            };
            if constexpr (kF8) {
#pragma unroll
                for (int grp = 0; grp < D / 64; ++grp) {
                    const uint4 h0 = lds128(kt + grp * 1024 + lane * 16);
                    const uint4 h1 = lds128(kt + grp * 1024 + 512 + lane * 16);
                    const uint32_t w0[4] = {h0.x, h0.y, h0.z, h0.w};
                    const uint32_t w1[4] = {h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const int kk = grp * 4 + s4;
                        uint32_t a[4];
                        e4m3x4_to_f16x2x2(w0[s4], a[0], a[2]);  // token g8
                        e4m3x4_to_f16x2x2(w1[s4], a[1], a[3]);  // token g8 + 8
#pragma unroll
                        for (int n = 0; n < NQ; ++n) {
                            uint32_t b0, b1;
                            q_frag(kk, n, b0, b1);
                            mma_16816_f16(sa[s4 & 1][n], a, b0, b1);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < C::kKS; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(kv_chunk_addr(kt, ka_tok, kk * 16 + ka_dof), a[0], a[1], a[2], a[3]);
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        uint32_t b0, b1;
                        q_frag(kk, n, b0, b1);
                        mma_16816(sa[kk & 1][n], a, b0, b1);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < NQ; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) sT[i][n][e] = sa[0][n][e] + sa[1][n][e];
        }

        // mask, scale to log2 units; element e of C is (token g8 + 8(e/2),
        // column 2cc + e%2)
        float sv[BPS][NQ][4];
        bool inside = true;
#pragma unroll
        for (int i = 0; i < BPS; ++i) {
            bool in = okb[i];
#pragma unroll
            for (int n = 0; n < NQ; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    in = in && (chi[n][e] == 0 ||
                                (base_tok[i] >= clo[n][e] && base_tok[i] + bs <= chi[n][e]));
            inside = inside && in;
        }
        if (__all_sync(0xffffffffu, inside)) {
#pragma unroll
            for (int i = 0; i < BPS; ++i)
#pragma unroll
                for (int n = 0; n < NQ; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sv[i][n][e] = sT[i][n][e] * p.scale_log2;
        } else {
#pragma unroll
            for (int i = 0; i < BPS; ++i)
#pragma unroll
                for (int n = 0; n < NQ; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int pos = base_tok[i] + g8 + 8 * (e >> 1);
                        const int lo = clo[n][e & 1], hi = chi[n][e & 1];
                        sv[i][n][e] = (okb[i] && pos >= lo && pos < hi)
                                          ? sT[i][n][e] * p.scale_log2
                                          : -INFINITY;
                    }
        }
        // column maxima: this lane's tokens, then the 8 lanes sharing cc
        float mu[NQ][2], al[NQ][2];
        bool grew = false;
#pragma unroll
        for (int n = 0; n < NQ; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < BPS; ++i) mx = fmaxf(mx, fmaxf(sv[i][n][e], sv[i][n][e + 2]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(mc[n][e], mx);
                mu[n][e] = mn == -INFINITY ? 0.f : mn;
                al[n][e] = fast_exp2(mc[n][e] - mu[n][e]);
                grew = grew || mn != mc[n][e];
                mc[n][e] = mn;
            }
        grew = __any_sync(0xffffffffu, grew);
        float pv[BPS][NQ][4];
#pragma unroll
        for (int n = 0; n < NQ; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < BPS; ++i) {
                    pv[i][n][e] = fast_exp2(sv[i][n][e] - mu[n][e]);
                    pv[i][n][e + 2] = fast_exp2(sv[i][n][e + 2] - mu[n][e]);
                    sum += pv[i][n][e] + pv[i][n][e + 2];
                }
                lc[n][e] = lc[n][e] * al[n][e] + sum;
            }
        if (grew) {
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    oT[mt][n][0] *= al[n][0];
                    oT[mt][n][1] *= al[n][1];
                    oT[mt][n][2] *= al[n][0];
                    oT[mt][n][3] *= al[n][1];
                }
        }

        // O^T += V^T P^T per block.  P as 16-bit pairs (token g8: columns
        // 2cc, 2cc+1) is row g8 of an 8x8 (tokens x columns) matrix;
        // movmatrix.trans hands each lane the (column g8: tokens 2cc, 2cc+1)
        // pair of the B fragment.  FP8: one f16 term (2^-11 relative).  bf16:
        // a bf16 pair hi + lo (lo = bf16(P - hi)), two products, so that P is
        // carried to about 2^-17 relative instead of the 2^-9 of one bf16
        // rounding.  Values of tokens outside every row's range are zeroed:
        // stale slots may hold anything, including NaN.
#pragma unroll
        for (int i = 0; i < BPS; ++i) {
            if (!okb[i]) continue;
            const uint32_t vt = stile + i * 2 * C::kTileBytes + C::kTileBytes;
            uint32_t pb[NQ][2], pl[NQ][2];
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                if constexpr (kF8) {
                    pb[n][0] = movmatrix_trans(pack_f16x2(pv[i][n][0], pv[i][n][1]));
                    pb[n][1] = movmatrix_trans(pack_f16x2(pv[i][n][2], pv[i][n][3]));
                } else {
                    const uint32_t h0 = pack_bf16x2(pv[i][n][0], pv[i][n][1]);
                    const uint32_t h1 = pack_bf16x2(pv[i][n][2], pv[i][n][3]);
                    const uint32_t l0 = pack_bf16x2(pv[i][n][0] - bf16lo_to_f32(h0),
                                                    pv[i][n][1] - bf16hi_to_f32(h0));
                    const uint32_t l1 = pack_bf16x2(pv[i][n][2] - bf16lo_to_f32(h1),
                                                    pv[i][n][3] - bf16hi_to_f32(h1));
                    pb[n][0] = movmatrix_trans(h0);
                    pb[n][1] = movmatrix_trans(h1);
                    pl[n][0] = movmatrix_trans(l0);
                    pl[n][1] = movmatrix_trans(l1);
                }
            }
            uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
            const int bt = base_tok[i];
            if (bt < lo_all || bt + bs > hi_all) {
                auto live = [&](int t) { return bt + t >= lo_all && bt + t < hi_all; };
                mk0 = (live(2 * cc) ? 0x0000ffffu : 0u) | (live(2 * cc + 1) ? 0xffff0000u : 0u);
                mk1 = (live(2 * cc + 8) ? 0x0000ffffu : 0u) | (live(2 * cc + 9) ? 0xffff0000u : 0u);
            }
            if constexpr (kF8) {
#pragma unroll
                for (int grp = 0; grp < D / 32; ++grp) {
                    const uint4 vw = lds128(vt + grp * 512 + lane * 16);
                    const uint32_t w4[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // m-tile 2grp + half: dims 16mt + g8 (word 2half) and
                        // 16mt + 8 + g8 (word 2half + 1)
                        uint32_t a[4];
                        e4m3x4_to_f16x2x2(w4[2 * half], a[0], a[2]);
                        e4m3x4_to_f16x2x2(w4[2 * half + 1], a[1], a[3]);
                        a[0] &= mk0;
                        a[1] &= mk0;
                        a[2] &= mk1;
                        a[3] &= mk1;
#pragma unroll
                        for (int n = 0; n < NQ; ++n)
                            mma_16816_f16(oT[2 * grp + half][n], a, pb[n][0], pb[n][1]);
                    }
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < C::kMT; ++mt) {
                    // a[0] (dim 16mt + g8, tokens 2cc, +1), a[1] (dim + 8),
                    // a[2], a[3]: the same for tokens 2cc + 8, +9
                    uint32_t a[4];
                    ldsm_x4_trans(kv_chunk_addr(vt, va_tok, mt * 16 + va_dof), a[0], a[1], a[2], a[3]);
                    a[0] &= mk0;
                    a[1] &= mk0;
                    a[2] &= mk1;
                    a[3] &= mk1;
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        mma_16816(oT[mt][n], a, pb[n][0], pb[n][1]);
                        mma_16816(oT[mt][n], a, pl[n][0], pl[n][1]);
                    }
                }
            }
        }

        // release the stage: its generic-proxy reads come before the next
        // async-proxy write into it
        fence_proxy_async_smem();
        __syncwarp();
        if (!prefix_item) {
            if (k + SPW < nk) issue(k + SPW);
        } else {
            if (lane == 0) mbar_arrive(&empty[st]);
            if (warp == 0 && k + STAGES < nk) {
                // every warp has released this stage before it is refilled
                bool freed = true;
                if (lane == 0) freed = mbar_wait(&empty[st], use & 1, p.wait_ns);
                if (!__shfl_sync(0xffffffffu, freed, 0)) {
                    // stop issuing: the passes after k still in flight land,
                    // then this warp leaves (the others run out of passes)
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                    drain(k + 1, k + STAGES);
                    break;
                }
                issue(k + STAGES);
            }
        }
    }

    // column sums over the 8 lanes sharing cc; FP8: the V scale on the values
#pragma unroll
    for (int n = 0; n < NQ; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            lc[n][e] += __shfl_xor_sync(0xffffffffu, lc[n][e], 4);
            lc[n][e] += __shfl_xor_sync(0xffffffffu, lc[n][e], 8);
            lc[n][e] += __shfl_xor_sync(0xffffffffu, lc[n][e], 16);
        }
    if constexpr (kF8) {
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
            for (int n = 0; n < NQ; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) oT[mt][n][e] *= p.v_scale;
    }

    // element e of oT[mt][n]: dim 16mt + g8 + 8(e/2), query row 8n + 2cc + e%2
    if (prefix_item) {
        // each warp owns its tile: write its rows directly
#pragma unroll
        for (int n = 0; n < NQ; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kq = tile * TR + 8 * n + 2 * cc + e;
                const int32_t pr = pair_row[kq];
                if (pr < 0) continue;
                const size_t pi = partial_index(p, pr, pair_head[kq], slot);
                float *dst = p.ws_o + pi * D + g8;
#pragma unroll
                for (int mt = 0; mt < C::kMT; ++mt) {
                    dst[16 * mt] = oT[mt][n][e];
                    dst[16 * mt + 8] = oT[mt][n][e + 2];
                }
                if (g8 == 0)
                    *reinterpret_cast<float2 *>(p.ws_ml + pi * 2) = make_float2(mc[n][e], lc[n][e]);
            }
        return;
    }
    // split item: this warp's rows of the one tile into the merge buffers
    __syncthreads();
#pragma unroll
    for (int n = 0; n < NQ; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = 8 * n + 2 * cc + e;
            if (row >= R) continue;
            float *dst = mbuf + (warp * R + row) * D + g8;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                dst[16 * mt] = oT[mt][n][e];
                dst[16 * mt + 8] = oT[mt][n][e + 2];
            }
            if (g8 == 0)
                *reinterpret_cast<float2 *>(mlbuf + (warp * R + row) * 2) =
                    make_float2(mc[n][e], lc[n][e]);
        }
    __syncthreads();
    for (int idx = threadIdx.x; idx < R * D; idx += NW * 32) {
        const int row = idx / D, d = idx % D;
        if (kMQ && row / G >= row_C) continue;  // no such query in this row
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mlbuf[(w * R + row) * 2]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float wgt = fast_exp2(mlbuf[(w * R + row) * 2] - M);
                acc += wgt * mbuf[(w * R + row) * D + d];
                lsum += wgt * mlbuf[(w * R + row) * 2 + 1];
            }
        }
        const size_t pi = kMQ ? partial_index(p, row_r, g * G + row % G, slot, row / G)
                              : partial_index(p, row_r, g * G + row, slot);
        p.ws_o[pi * D + d] = acc;
        if (d == 0) *reinterpret_cast<float2 *>(p.ws_ml + pi * 2) = make_float2(M, lsum);
    }
}

template <int D, bool kMQ, bool kF8, int NQ>
__global__ void __launch_bounds__(kDecodeWarps * 32, KvCfg<D, kF8, NQ>::kCtasPerSm)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p)
{
    decode_split_body<D, kMQ, kF8, NQ>(kmap, vmap, p, blockIdx.x);
}

// Several decode calls in one launch (groups of a model's layers that share
// the head shape, e.g. a full-attention group and a sliding group): CTAs
// [cta_end[i-1], cta_end[i]) do group i's work.
template <int D, bool kF8, int NQ>
__global__ void __launch_bounds__(kDecodeWarps * 32, KvCfg<D, kF8, NQ>::kCtasPerSm)
    decode_split_grouped_kernel(const __grid_constant__ GroupedDecode gd)
{
    int i = 0;
    const int64_t b = blockIdx.x;
    while (i + 1 < gd.n && b >= gd.cta_end[i]) ++i;
    const int64_t first = i > 0 ? gd.cta_end[i - 1] : 0;
    decode_split_body<D, false, kF8, NQ>(gd.kmap[i], gd.vmap[i], gd.g[i], b - first);
}

template <int D, bool kF8, int NQ = 1>
static cudaError_t launch_split_grouped(const GroupedDecode &gd, cudaStream_t stream)
{
    const int64_t ctas = gd.cta_end[gd.n - 1];
    if (ctas == 0) return cudaSuccess;
    auto kern = decode_split_grouped_kernel<D, kF8, NQ>;
    const int smem = KvSmem<D, kF8, NQ>::kLaunchBytes;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_DECODE_SPLIT, stream);
    err = launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(kDecodeWarps * 32), smem, stream, gd);
    prof_end(PKV_KERNEL_DECODE_SPLIT, stream);
    return err;
}

template <int D, bool kMQ, bool kF8, int NQ = 1>
static cudaError_t launch_split(const DecodeParams &p, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, cudaStream_t stream)
{
    const int64_t ctas = p.plan.n_prefix_ctas + p.plan.n_suffix_ctas;
    if (ctas == 0) return cudaSuccess;
    auto kern = decode_split_kernel<D, kMQ, kF8, NQ>;
    const int smem = KvSmem<D, kF8, NQ>::kLaunchBytes;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    // the largest shared-memory carveout, so that kCtasPerSm CTAs are resident per SM
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_DECODE_SPLIT, stream);
    err = launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(kDecodeWarps * 32), smem,
                     stream, kmap, vmap, p);
    prof_end(PKV_KERNEL_DECODE_SPLIT, stream);
    return err;
}

}  // namespace pkv
