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
//       16-row query tile holds the G q heads of (r, g).
// K and V (block, kv head) tiles are brought into shared memory with one TMA
// tensor load each (5-D maps viewing [block][kv head][slot][dim] as
// (64 dims, slot, 64-dim region, kv head, block), 128-byte swizzle, so a tile
// lands as one 2 KiB swizzled region per 64 dims) that completes on an mbarrier.
//   split item: each of the four warps takes every fourth block of the run and
//       keeps its own ring of stages: it issues the loads of its next blocks
//       itself as it frees a stage, so no warp ever waits behind another;
//   prefix item: the four warps share one ring (each owns a query tile and
//       reads every block); warp 0 refills a stage once all four released it.
// Warps compute S = Q K^T and O += P V with mma.sync m16n8k16 (fp32
// accumulate): M = 16 query rows, N = 8 tokens or 8 dims.  The online softmax
// runs on the accumulator fragments with quad shuffles.  Each tile's partial
// (max in log2 units, sum, unnormalised O) goes to the workspace.
//   bf16 pools: bf16 operands; P enters the P.V product as two bf16 terms
//       (hi + lo) so that its rounding stays far below the output's own bf16
//       rounding.
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

template <int D, bool kF8>
struct KvCfg {
    static constexpr int kTok = 16;                       // block_size
    static constexpr int kElem = kF8 ? 1 : 2;             // bytes per K/V element
    static constexpr int kTileBytes = kTok * D * kElem;   // one (block, kv head) tile of K or V
    static constexpr int kStageBytes = 2 * kTileBytes;    // K + V
    // query fragments stay in registers for head_dim <= 128; there the query
    // tiles are staged through the ring before the first load, otherwise they
    // keep a region of their own
    static constexpr bool kQInRegs = D <= 128;
    static constexpr int kTiles = 4;                      // query tiles of a prefix item
    // ring sized so that two CTAs fit on an SM
    static constexpr int kRingBytes = (D == 256 ? 64 : 96) * 1024;
    static constexpr int kStages = kRingBytes / kStageBytes;
    static constexpr int kStagesPerWarp = kStages / kDecodeWarps;  // split items
    static_assert(kStages % kDecodeWarps == 0, "split items give each warp the same stages");
    static constexpr int kRegions = D / 64;               // 64-dim swizzled regions per tile
    static constexpr int kRegionBytes = kTok * 128;
    static constexpr int kQStride = (D + 8) * 2;          // padded query row (bytes)
    static constexpr int kQTileBytes = 16 * kQStride;
    static constexpr int kNT = D / 8;                     // 8-dim output n-tiles
    static constexpr int kKS = D / 16;                    // 16-dim k-steps of Q K^T
};

template <int D, bool kF8>
struct KvSmem {
    using C = KvCfg<D, kF8>;
    static constexpr int kStageOff = 0;
    static constexpr int kQOff = C::kQInRegs ? 0 : C::kRingBytes;
    static constexpr int kBarOff =
        C::kQInRegs ? C::kRingBytes : C::kRingBytes + C::kTiles * C::kQTileBytes;
    static constexpr int kOkOff = kBarOff + 2 * C::kStages * 8;
    static constexpr int kPairOff = kOkOff + C::kStages * 4;
    static constexpr int kMiscOff = kPairOff + 3 * C::kTiles * 16 * 4;
    static constexpr int kBytes = kMiscOff + 16;
    static constexpr int kLaunchBytes = kBytes + 1024;  // room to align the base to 1024
    static_assert(C::kTiles * C::kQTileBytes <= C::kRingBytes || !C::kQInRegs,
                  "query tiles staged through the ring fit in it");
    static_assert(kDecodeWarps * 16 * D * 4 + kDecodeWarps * 16 * 8 <= kBarOff,
                  "the merge buffers fit below the barriers");
};

// Swizzled shared address of the 16-byte chunk holding dims d0..d0+7 of token
// `tok` in a K/V tile (TMA SWIZZLE_128B: chunk index XOR (line % 8)).
template <int D>
__device__ __forceinline__ uint32_t kv_chunk_addr(uint32_t tile, int tok, int d0)
{
    return tile + (d0 >> 6) * KvCfg<D, false>::kRegionBytes + tok * 128 +
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

template <int D, bool kMQ, bool kF8>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p)
{
    using C = KvCfg<D, kF8>;
    using SM = KvSmem<D, kF8>;
    constexpr int NW = kDecodeWarps;
    constexpr int STAGES = C::kStages;
    constexpr int SPW = C::kStagesPerWarp;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stage_mem = smem + SM::kStageOff;
    uint8_t *q_mem = smem + SM::kQOff;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::kBarOff);
    uint64_t *empty = full + STAGES;
    int32_t *stage_ok = reinterpret_cast<int32_t *>(smem + SM::kOkOff);
    int32_t *pair_row = reinterpret_cast<int32_t *>(smem + SM::kPairOff);
    int32_t *pair_head = pair_row + C::kTiles * 16;
    int32_t *pair_len = pair_head + C::kTiles * 16;
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
    const bool prefix_item = static_cast<int64_t>(blockIdx.x) < p.plan.n_prefix_ctas;
    int32_t b0, nblk, slot, tab_row, g, lo_all, hi_all, tiles;
    // split item only: the row, its query count and first packed query
    int32_t row_r = 0, row_C = 1, row_q0 = 0;
    // M-rows of a split item: the G heads of one query (decode), or (query,
    // head) pairs of a row's few queries (kMQ: a verify step)
    const int R = kMQ ? G * p.max_q : G;
    if (!prefix_item) {
        int64_t bid = static_cast<int64_t>(blockIdx.x) - p.plan.n_prefix_ctas;
        const int32_t s = static_cast<int32_t>(bid % p.plan.n_suffix_splits);
        bid /= p.plan.n_suffix_splits;
        g = static_cast<int32_t>(bid % p.hkv);
        row_r = static_cast<int32_t>(bid / p.hkv);
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
    } else {
        tiles = C::kTiles;
        int64_t bid = blockIdx.x;
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
        for (int i = threadIdx.x; i < tiles * 16; i += blockDim.x) pair_row[i] = -1;
        __syncthreads();
        if (warp == 0) {
            // rows of the group in ascending order; pair k = rank * G + j
            const int32_t per_cta = tiles * 16;
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
        for (int i = threadIdx.x; i < tiles * 16 * nblk; i += blockDim.x) {
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
        for (int i = threadIdx.x; i < tiles * 16 * kVec; i += blockDim.x) {
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
            *reinterpret_cast<uint4 *>(q_mem + (row / 16) * C::kQTileBytes +
                                       (row % 16) * C::kQStride + v * 16) = val;
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
    const uint32_t q_lane = smem_u32(q_mem + tile * C::kQTileBytes) +
                            (((lane >> 3) & 1) * 8 + (lane & 7)) * C::kQStride + (lane >> 4) * 16;
    uint32_t qf[C::kQInRegs ? C::kKS : 1][4];
    if constexpr (C::kQInRegs) {
#pragma unroll
        for (int kk = 0; kk < C::kKS; ++kk)
            ldsm_x4(q_lane + kk * 32, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
        // the ring is about to be overwritten by TMA (async proxy) after these
        // generic-proxy reads and writes of the staged query tiles
        fence_proxy_async_smem();
        __syncthreads();
    }

    // ------------------------------------------------------------- loads
    // split item: warp w's blocks are b0 + w + NW*k (k = 0 .. nk-1); its use k
    // goes to stage w*SPW + k % SPW.  prefix item: block k to stage k % STAGES,
    // loads issued by warp 0.
    const uint64_t policy = l2_evict_first_policy();
    const int32_t *table_row = p.tables + static_cast<int64_t>(tab_row) * p.width + b0;
    const int32_t nk = prefix_item ? nblk : (nblk > warp ? (nblk - warp + NW - 1) / NW : 0);
    const bool issuer = !prefix_item || warp == 0;
    BlockIds ids;
    if (issuer) ids.init(table_row, prefix_item ? 0 : warp, prefix_item ? 1 : NW, nk, lane);
    auto stage_of = [&](int32_t k) { return prefix_item ? k % STAGES : warp * SPW + k % SPW; };
    auto issue = [&](int32_t k) {  // whole warp; lane 0 issues
        const int32_t bj = ids.next(k, lane);
        if (lane == 0) {
            const int st = stage_of(k);
            const bool ok = static_cast<uint32_t>(bj) < static_cast<uint32_t>(p.num_blocks);
            stage_ok[st] = ok ? 1 : 0;
            if (ok) {
                mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                uint8_t *kdst = stage_mem + st * C::kStageBytes;
                uint8_t *vdst = kdst + C::kTileBytes;
                if constexpr (kF8) {
                    // the tile is one contiguous run of the pool
                    const int64_t off = (static_cast<int64_t>(bj) * p.hkv + g) * C::kTileBytes;
                    bulk_load(kdst, static_cast<const uint8_t *>(p.k_pool) + off, C::kTileBytes,
                              &full[st], policy);
                    bulk_load(vdst, static_cast<const uint8_t *>(p.v_pool) + off, C::kTileBytes,
                              &full[st], policy);
                } else {
                    // one box per (block, kv head) tile: every 64-dim region at once
                    tma_load_5d(kdst, &kmap, &full[st], 0, 0, 0, g, bj, policy);
                    tma_load_5d(vdst, &vmap, &full[st], 0, 0, 0, g, bj, policy);
                }
            } else {
                report(p.status, PKV_DEV_BAD_BLOCK);
                mbar_arrive(&full[st]);
            }
        }
    };
    const int32_t depth = prefix_item ? STAGES : SPW;
    if (issuer)
        for (int32_t k = 0; k < min(depth, nk); ++k) issue(k);

    // ---------------------------------------------------------------- compute
    const int qd = lane >> 2;        // fragment rows qd and qd + 8
    const int c2 = 2 * (lane & 3);   // fragment columns c2, c2 + 1
    int lo0, hi0, lo1, hi1;
    if (!prefix_item) {
        if constexpr (kMQ) {
            // query t of the row sits at L - C + t: causal limit hi, window start lo
            auto limits = [&](int row, int &lo, int &hi) {
                const int t = row / G;
                hi = (row < R && t < row_C) ? hi_all - row_C + t + 1 : 0;
                lo = (p.window > 0 && hi > 0) ? max(0, hi - p.window) : 0;
            };
            limits(qd, lo0, hi0);
            limits(qd + 8, lo1, hi1);
        } else {
            lo0 = lo1 = lo_all;
            hi0 = hi1 = hi_all;
        }
    } else {
        lo0 = lo1 = 0;
        const int k0 = tile * 16 + qd;
        hi0 = pair_row[k0] >= 0 ? pair_len[k0] : 0;
        hi1 = pair_row[k0 + 8] >= 0 ? pair_len[k0 + 8] : 0;
    }

    float o[C::kNT][4];
#pragma unroll
    for (int nt = 0; nt < C::kNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // lane-constant parts of the ldmatrix addresses
    const int k_tok = (lane >> 4) * 8 + (lane & 7);
    const int k_dof = ((lane >> 3) & 1) * 8;
    const int v_tok = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int v_dof = (lane >> 4) * 8;

    for (int32_t k = 0; k < nk; ++k) {
        const int st = stage_of(k);
        const int32_t use = prefix_item ? k / STAGES : k / SPW;
        const bool got = mbar_wait(&full[st], use & 1);
        if (__any_sync(0xffffffffu, !got)) {
            if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
            break;
        }
        const bool ok = stage_ok[st] != 0;
        const uint32_t kt = smem_u32(stage_mem + st * C::kStageBytes);
        const uint32_t vt = kt + C::kTileBytes;
        const int base_tok = (b0 + (prefix_item ? k : warp + NW * k)) * bs;

        // S = Q K^T  (16 rows x 16 tokens)
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if constexpr (kF8) {
            // lane's 16 bytes of a (64-dim group, token half) hold its B
            // fragments of the group's four 16-dim steps
#pragma unroll
            for (int grp = 0; grp < D / 64; ++grp)
#pragma unroll
                for (int jt = 0; jt < 2; ++jt) {
                    const uint4 kw = lds128(kt + grp * 1024 + jt * 512 + lane * 16);
                    const uint32_t w4[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const int kk = grp * 4 + s4;
                        uint32_t a[4];
                        if constexpr (C::kQInRegs) {
                            a[0] = qf[kk][0]; a[1] = qf[kk][1]; a[2] = qf[kk][2]; a[3] = qf[kk][3];
                        } else {
                            ldsm_x4(q_lane + kk * 32, a[0], a[1], a[2], a[3]);
                        }
                        uint32_t b0, b1;
                        e4m3x4_to_f16x2x2(w4[s4], b0, b1);
                        mma_16816_f16(sacc[jt], a, b0, b1);
                    }
                }
        } else {
#pragma unroll
            for (int kk = 0; kk < C::kKS; ++kk) {
                uint32_t a[4];
                if constexpr (C::kQInRegs) {
                    a[0] = qf[kk][0]; a[1] = qf[kk][1]; a[2] = qf[kk][2]; a[3] = qf[kk][3];
                } else {
                    ldsm_x4(q_lane + kk * 32, a[0], a[1], a[2], a[3]);
                }
                uint32_t k0, k1, k2, k3;
                ldsm_x4(kv_chunk_addr<D>(kt, k_tok, kk * 16 + k_dof), k0, k1, k2, k3);
                mma_16816(sacc[0], a, k0, k1);
                mma_16816(sacc[1], a, k2, k3);
            }
        }

        // mask, scale to log2 units, online softmax over the quad's row
        float s[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int pos = base_tok + j * 8 + c2 + (e & 1);
                const int lo = e < 2 ? lo0 : lo1, hi = e < 2 ? hi0 : hi1;
                s[j][e] = (ok && pos >= lo && pos < hi) ? sacc[j][e] * p.scale_log2 : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        // P = 2^(s - m) as a bf16 pair hi + lo (lo = bf16(P - hi)): the P.V
        // product then carries P to about 2^-17 relative instead of the 2^-9
        // of a single bf16 rounding
        float pf[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pf[j][0] = fast_exp2(s[j][0] - mu0);
            pf[j][1] = fast_exp2(s[j][1] - mu0);
            pf[j][2] = fast_exp2(s[j][2] - mu1);
            pf[j][3] = fast_exp2(s[j][3] - mu1);
        }
        uint32_t pa[4], pl[4];
        if constexpr (kF8) {
            pa[0] = pack_f16x2(pf[0][0], pf[0][1]);
            pa[1] = pack_f16x2(pf[0][2], pf[0][3]);
            pa[2] = pack_f16x2(pf[1][0], pf[1][1]);
            pa[3] = pack_f16x2(pf[1][2], pf[1][3]);
        } else {
            pa[0] = pack_bf16x2(pf[0][0], pf[0][1]);
            pa[1] = pack_bf16x2(pf[0][2], pf[0][3]);
            pa[2] = pack_bf16x2(pf[1][0], pf[1][1]);
            pa[3] = pack_bf16x2(pf[1][2], pf[1][3]);
            pl[0] = pack_bf16x2(pf[0][0] - bf16lo_to_f32(pa[0]), pf[0][1] - bf16hi_to_f32(pa[0]));
            pl[1] = pack_bf16x2(pf[0][2] - bf16lo_to_f32(pa[1]), pf[0][3] - bf16hi_to_f32(pa[1]));
            pl[2] = pack_bf16x2(pf[1][0] - bf16lo_to_f32(pa[2]), pf[1][1] - bf16hi_to_f32(pa[2]));
            pl[3] = pack_bf16x2(pf[1][2] - bf16lo_to_f32(pa[3]), pf[1][3] - bf16hi_to_f32(pa[3]));
        }
        l0 = l0 * al0 + ((pf[0][0] + pf[0][1]) + (pf[1][0] + pf[1][1]));
        l1 = l1 * al1 + ((pf[0][2] + pf[0][3]) + (pf[1][2] + pf[1][3]));
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) {
            o[nt][0] *= al0;
            o[nt][1] *= al0;
            o[nt][2] *= al1;
            o[nt][3] *= al1;
        }

        // O += P V  (values of tokens outside every row's range are zeroed:
        // stale slots may hold anything, including NaN)
        if (ok) {
            uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
            if (base_tok < lo_all || base_tok + bs > hi_all) {
                auto live = [&](int t) {
                    return base_tok + t >= lo_all && base_tok + t < hi_all;
                };
                mk0 = (live(c2) ? 0x0000ffffu : 0u) | (live(c2 + 1) ? 0xffff0000u : 0u);
                mk1 = (live(c2 + 8) ? 0x0000ffffu : 0u) | (live(c2 + 9) ? 0xffff0000u : 0u);
            }
            if constexpr (kF8) {
                // lane's 16 bytes of a 32-dim group hold its B fragments of
                // the group's four 8-dim n-tiles
#pragma unroll
                for (int grp = 0; grp < D / 32; ++grp) {
                    const uint4 vw = lds128(vt + grp * 512 + lane * 16);
                    const uint32_t w4[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
                    for (int jn = 0; jn < 4; ++jn) {
                        uint32_t b0, b1;
                        e4m3x4_to_f16x2x2(w4[jn], b0, b1);
                        mma_16816_f16(o[grp * 4 + jn], pa, b0 & mk0, b1 & mk1);
                    }
                }
            } else {
#pragma unroll
                for (int np = 0; np < C::kNT / 2; ++np) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_trans(kv_chunk_addr<D>(vt, v_tok, np * 16 + v_dof), v0, v1, v2, v3);
                    v0 &= mk0; v1 &= mk1; v2 &= mk0; v3 &= mk1;
                    mma_16816(o[2 * np], pa, v0, v1);
                    mma_16816(o[2 * np + 1], pa, v2, v3);
                    mma_16816(o[2 * np], pl, v0, v1);
                    mma_16816(o[2 * np + 1], pl, v2, v3);
                }
            }
        }

        // release the stage: its generic-proxy reads come before the next
        // TMA write into it
        fence_proxy_async_smem();
        __syncwarp();
        if (!prefix_item) {
            if (k + SPW < nk) issue(k + SPW);
        } else {
            if (lane == 0) mbar_arrive(&empty[st]);
            if (warp == 0 && k + STAGES < nk) {
                // every warp has released this stage before it is refilled
                bool freed = true;
                if (lane == 0) freed = mbar_wait(&empty[st], use & 1);
                if (!__shfl_sync(0xffffffffu, freed, 0)) {
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                } else {
                    issue(k + STAGES);
                }
            }
        }
    }

    if constexpr (kF8) {
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) {
            o[nt][0] *= p.v_scale;
            o[nt][1] *= p.v_scale;
            o[nt][2] *= p.v_scale;
            o[nt][3] *= p.v_scale;
        }
    }

    // row sums: the quad's four partial sums
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    if (prefix_item) {
        // each warp owns its tile: write its rows directly
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int k = tile * 16 + qd + half * 8;
            const int32_t pr = pair_row[k];
            if (pr < 0) continue;
            const size_t pi = partial_index(p, pr, pair_head[k], slot);
            float *dst = p.ws_o + pi * D;
#pragma unroll
            for (int nt = 0; nt < C::kNT; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8 + c2) =
                    make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
            if ((lane & 3) == 0)
                *reinterpret_cast<float2 *>(p.ws_ml + pi * 2) =
                    make_float2(half ? m1 : m0, half ? l1 : l0);
        }
        return;
    }

    // split item: merge the four warps' partials of the one tile through
    // shared memory (the ring is free once every warp is past its last block)
    float *mbuf = reinterpret_cast<float *>(stage_mem);  // [NW][R][D]
    float *mlbuf = mbuf + NW * 16 * D;                    // [NW][R][2], R <= 16
    __syncthreads();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int row = qd + half * 8;
        if (row >= R) continue;
        float *dst = mbuf + (warp * R + row) * D;
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt)
            *reinterpret_cast<float2 *>(dst + nt * 8 + c2) =
                make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
        if ((lane & 3) == 0)
            *reinterpret_cast<float2 *>(mlbuf + (warp * R + row) * 2) =
                make_float2(half ? m1 : m0, half ? l1 : l0);
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

template <int D, bool kMQ, bool kF8>
static cudaError_t launch_split(const DecodeParams &p, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, cudaStream_t stream)
{
    const int64_t ctas = p.plan.n_prefix_ctas + p.plan.n_suffix_ctas;
    if (ctas == 0) return cudaSuccess;
    auto kern = decode_split_kernel<D, kMQ, kF8>;
    const int smem = KvSmem<D, kF8>::kLaunchBytes;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    // the largest shared-memory carveout, so that two CTAs are resident per SM
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
