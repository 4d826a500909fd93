// Chunked prefill against a paged prefix ("perf.md", gather_kv_for_prefill_chunk:
// a prefill chunk attends its cached prefix through the pages; "paged-cache.md":
// chunk boundaries change the reduction order, not the result).  Query i of a
// row's chunk sits at absolute position p = L - C + i and attends positions
// max(0, p - W + 1) .. p: the whole prefix and the chunk causally.
//
// bf16 kernel, one CTA per (row, kv head, two tiles of 128/G queries).  A
// tile's 128 M-rows are (query, head) pairs of all G q heads of the kv head,
// and both tiles share every K/V tile, so K/V are loaded once per 256 query
// rows.  QK^T and PV are dense contractions and run on the 5th-generation
// tensor cores:
//   warps 0/2 TMA producers: K and V tiles of 128 keys (8 paged blocks, two
//             64-dim boxes each) into 2-stage rings; a K stage is freed once
//             both S products are computed, a V stage once both P.V are;
//   warp 1    allocates tensor memory and issues tcgen05.mma from one elected
//             lane: S_x = Q_x K^T into tensor memory (both operands K-major,
//             128-byte swizzle), then O_x += P_x V with P read from tensor
//             memory (V MN-major), in the order PV_A(j), S_A(j+1), PV_B(j),
//             S_B(j+1);
//   warps 4-7 / 8-11  softmax of tile A / tile B, concurrently, one M-row per
//             thread: S from tensor memory, causal / window / range mask,
//             running max kept within 2^8 of the true maximum (O is rescaled
//             in tensor memory only when it moves further), P written back over
//             S as bf16 hi + lo terms, 8 columns each per 16 keys (P.V then carries P to
//             ~2^-17 relative), and the epilogue O / l to global memory.
//             S is read twice from tensor memory (row maximum, then P), which
//             keeps a thread's live scores to 32 at a time.
// f32 kernel: CUDA cores, the same work split with 16 (query, head) pairs per
// CTA, for the fp32 pools.
#include "decode_common.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace pf {
constexpr int kD = 128;
constexpr int kRows = 128;                // M of one query tile
constexpr int kQTiles = 2;                // query tiles per CTA, sharing every K/V tile
constexpr int kKeys = 128;                // keys per K/V tile (8 blocks of 16)
constexpr int kQBytes = kRows * 2 * 128;  // one query tile: two 64-dim swizzled regions
constexpr int kKVRegion = kKeys * 128;    // 16 KiB
constexpr int kTileBytes = 2 * kKVRegion; // 32 KiB: a K or a V tile
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQTiles * kQBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
// barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[A,B], p_full[A,B], pv_done[A,B]
constexpr int kNumBars = 14;
constexpr int kMaskOff = kBarOff + kNumBars * 8;
constexpr int kTmemOff = kMaskOff + kKStages * 4;
constexpr int kBytes = kTmemOff + 16;
constexpr int kLaunchBytes = kBytes + 1024;
// warps: 0 K producer, 1 MMA issue, 2 V producer, 3 idle (warpgroup 0);
// 4-7 softmax of query tile A, 8-11 of tile B (one M-row per thread)
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;       // S_A, S_B, O_A, O_B
constexpr uint32_t kRescaleLog2 = 8;      // O is rescaled only when the max grows past 2^8
static_assert(kLaunchBytes <= 227 * 1024, "shared memory of one CTA");
}  // namespace pf

struct PrefillRowInfo {
    int32_t r, g, i0, nq, L, C, kv_lo, kv_hi;
};

__device__ __forceinline__ bool prefill_item(const PrefillParams &p, int64_t bid, int qpc,
                                             PrefillRowInfo &w)
{
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

// Wait by one lane, result broadcast to the warp; reports a timeout.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int lane, int32_t *status)
{
    bool ok = true;
    if (lane == 0) ok = mbar_wait(bar, parity);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) report(status, PKV_DEV_TIMEOUT);
    return ok;
}

// ---------------------------------------------------------------------------
// bf16, tcgen05
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(pf::kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const PrefillParams p)
{
    using namespace pf;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *q_s = smem + kQOff;
    uint8_t *k_s = smem + kKOff;
    uint8_t *v_s = smem + kVOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *k_full = bars, *k_empty = bars + 2, *v_full = bars + 4, *v_empty = bars + 6,
             *s_full = bars + 8, *p_full = bars + 10, *pv_done = bars + 12;
    uint32_t *kmask = reinterpret_cast<uint32_t *>(smem + kMaskOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTmemOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int qpt = kRows / G;  // queries per query tile

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    pdl_wait();
    pdl_trigger();

    PrefillRowInfo w;
    if (!prefill_item(p, blockIdx.x, kQTiles * qpt, w)) return;
    const int32_t jt0 = w.kv_lo / kKeys;
    const int32_t ntile = (w.kv_hi - 1) / kKeys - jt0 + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1 + kSoftmaxWarps);  // both S products + the kmask reads
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kSoftmaxWarps / kQTiles);
            mbar_init(&pv_done[i], 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(tmem_slot, kTmemCols);

    // query tiles: tile x row i = (query t = x * qpt + i / G, head h = i % G);
    // the 256 softmax threads load one row each
    if (warp >= 4) {
        const int ii = threadIdx.x - 128;
        const int x = ii / kRows, i = ii % kRows;
        const int t = x * qpt + i / G, h = i % G;
        const bool valid = i < qpt * G && t < w.nq;
        const uint4 *src = reinterpret_cast<const uint4 *>(p.q) +
                           ((static_cast<int64_t>(__ldg(p.cu_q_lens + w.r)) + w.i0 + t) * p.hq +
                            w.g * G + h) * (kD / 8);
        uint8_t *qt_s = q_s + x * kQBytes;
        // a negative scale: stage -q (sign bits flipped, exact), so that the
        // scores the tensor cores produce always take a positive factor
        const uint32_t flip = p.scale_log2 < 0.f ? 0x80008000u : 0u;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            v.x ^= flip;
            v.y ^= flip;
            v.z ^= flip;
            v.w ^= flip;
            *reinterpret_cast<uint4 *>(qt_s + (c >> 3) * (kRows * 128) + i * 128 +
                                       (((c & 7) ^ (i & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();  // read by the tensor cores (async proxy)
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    // tensor memory: S_x at columns 128x, O_x at 256 + 128x
    auto tS = [&](int x) { return tmem + 128u * static_cast<uint32_t>(x); };
    auto tO = [&](int x) { return tmem + 256u + 128u * static_cast<uint32_t>(x); };

    if (warp < 4) {
      if (warp == 0 || warp == 2) {
        // ------------------------------------------ K (warp 0) / V (warp 2) producer
        const bool is_k = warp == 0;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        uint8_t *ring = is_k ? k_s : v_s;
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *empty = is_k ? k_empty : v_empty;
        const uint64_t policy = l2_evict_last_policy();  // re-read by the row's other CTAs
        const int32_t *trow = p.tables + static_cast<int64_t>(w.r) * p.width;
        for (int32_t jj = 0; jj < ntile; ++jj) {
            const int st = jj & 1;
            if (jj >= 2 && !warp_wait(&empty[st], ((jj >> 1) + 1) & 1, lane, p.status)) break;
            const int32_t kb = (jt0 + jj) * (kKeys / 16) + lane;  // logical block of lane < 8
            const bool in_range = lane < 8 && kb < p.width && kb * 16 < w.kv_hi &&
                                  (kb + 1) * 16 > w.kv_lo;
            const int32_t id = in_range ? __ldg(trow + kb) : -1;
            const bool good = in_range && static_cast<uint32_t>(id) < static_cast<uint32_t>(p.num_blocks);
            if (is_k && in_range && !good) report(p.status, PKV_DEV_BAD_BLOCK);
            const uint32_t mask = __ballot_sync(0xffffffffu, good) & 0xffu;
            if (lane == 0) {
                if (is_k) kmask[st] = mask;
                if (mask == 0)
                    mbar_arrive(&full[st]);
                else
                    mbar_arrive_expect_tx(&full[st], __popc(mask) * 2 * 2048);
            }
            __syncwarp();
            uint8_t *dst = ring + st * kTileBytes;
            for (int b = 0; b < 8; ++b) {
                const int32_t bid = __shfl_sync(0xffffffffu, id, b);
                if (((mask >> b) & 1u) && elect_one()) {
                    tma_load_4d(dst + b * 2048, map, &full[st], 0, 0, w.g, bid, policy);
                    tma_load_4d(dst + kKVRegion + b * 2048, map, &full[st], 64, 0, w.g, bid, policy);
                }
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        // Order per K/V tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while
        // one tile's warpgroup turns S into P the tensor cores work for the
        // other.  The tensor cores execute in issue order, so S_x(j+1)
        // completing also means PV_x(j) is done.
        constexpr uint32_t idS = tc::idesc_bf16(kRows, kKeys, 0, 0);
        constexpr uint32_t idO = tc::idesc_bf16(kRows, kD, 0, 1);
        // Descriptors are built once: a single issuing thread that rebuilds
        // them per instruction spends longer than the tensor cores take for
        // an N=128 product.  Moving along K (or to the next 16 keys of V)
        // adds the byte offset / 16 to the start-address field, which cannot
        // carry out of it inside shared memory.
        const uint64_t dq0 = tc::smem_desc(smem_u32(q_s), 16, 1024);
        const uint64_t dq1 = tc::smem_desc(smem_u32(q_s + kQBytes), 16, 1024);
        const uint64_t dk0 = tc::smem_desc(smem_u32(k_s), 16, 1024);
        const uint64_t dk1 = tc::smem_desc(smem_u32(k_s + kTileBytes), 16, 1024);
        const uint64_t dv0 = tc::smem_desc(smem_u32(v_s), kKVRegion, 1024);
        const uint64_t dv1 = tc::smem_desc(smem_u32(v_s + kTileBytes), kKVRegion, 1024);
        // The whole warp runs these; one elected lane issues each product
        // and the commits (an issuing thread inside a lane-0 branch is
        // measurably slower to issue).
        auto s_mma = [&](int x, int32_t jj) {
            const uint64_t qd = x ? dq1 : dq0, kd = (jj & 1) ? dk1 : dk0;
            const uint32_t d = tS(x);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kKVRegion + (kk & 3) * 32) >> 4);
                if (elect_one()) tc::mma_ss(d, qd + off, kd + off, idS, kk > 0 ? 1u : 0u);
            }
            if (elect_one()) tc::commit(&s_full[x]);
            __syncwarp();
        };
        auto pv_mma = [&](int x, int32_t jj) {
            const uint64_t vd = (jj & 1) ? dv1 : dv0;
            const uint32_t d = tO(x), a = tS(x);
            const uint32_t first = jj > 0 ? 1u : 0u;
            // keys 16g..16g+15 hold P hi in S columns 16g..16g+7 and P lo in
            // 16g+8..16g+15 (bf16 pairs)
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    if (elect_one())
                        tc::mma_ts(d, a + 16 * kk + 8 * part,
                                   vd + static_cast<uint64_t>(kk * 2048 >> 4), idO,
                                   (part > 0 || kk > 0) ? 1u : first);
            if (elect_one()) tc::commit(&pv_done[x]);
            __syncwarp();
        };
        bool ok = warp_wait(&k_full[0], 0, lane, p.status);
        if (ok) {
            tc::fence_after();
            s_mma(0, 0);
            s_mma(1, 0);
            if (elect_one()) tc::commit(&k_empty[0]);
            __syncwarp();
        }
        for (int32_t jj = 0; jj < ntile && ok; ++jj) {
            const bool more = jj + 1 < ntile;
            ok = warp_wait(&p_full[0], jj & 1, lane, p.status) &&
                 warp_wait(&v_full[jj & 1], (jj >> 1) & 1, lane, p.status);
            if (!ok) break;
            tc::fence_after();
            pv_mma(0, jj);
            if (more) {
                ok = warp_wait(&k_full[(jj + 1) & 1], ((jj + 1) >> 1) & 1, lane, p.status);
                if (!ok) break;
                tc::fence_after();
                s_mma(0, jj + 1);
            }
            ok = warp_wait(&p_full[1], jj & 1, lane, p.status);
            if (!ok) break;
            tc::fence_after();
            pv_mma(1, jj);
            if (elect_one()) tc::commit(&v_empty[jj & 1]);
            __syncwarp();
            if (more) {
                s_mma(1, jj + 1);
                if (elect_one()) tc::commit(&k_empty[(jj + 1) & 1]);
                __syncwarp();
            }
        }
      }
    } else {
        // ------------------------------------------------------------ softmax
        // warpgroup x (warps 4-7: tile A, 8-11: tile B), one M-row per thread:
        // tensor-memory lane quarter warp % 4, all 128 key columns of S
        const int x = (warp >> 2) - 1;
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const int row = 32 * (warp & 3) + lane;
        const int t = x * qpt + row / G;
        const bool valid_row = row < qpt * G && t < w.nq;
        const int32_t qpos = w.L - w.C + w.i0 + t;
        const int32_t qlo = p.window > 0 ? max(0, qpos - p.window + 1) : 0;
        const uint32_t sx = tS(x) + lane_base, ox = tO(x) + lane_base;
        // |scale| * log2(e) (q was staged negated for a negative scale), kept
        // away from 0 so that a masked score (-inf) never meets a zero factor
        const float sl = fmaxf(fabsf(p.scale_log2), 1e-30f);
        float m_ref = -INFINITY, l = 0.f;
        bool abort = false;
        for (int32_t jj = 0; jj < ntile; ++jj) {
            const int ks = jj & 1;
            const int32_t tbase = (jt0 + jj) * kKeys;
            bool got = mbar_wait(&s_full[x], jj & 1);
            got = got && mbar_wait(&k_full[ks], (jj >> 1) & 1);  // for kmask
            if (__any_sync(0xffffffffu, !got)) {
                if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                abort = true;
                break;
            }
            const uint32_t mask = kmask[ks];
            __syncwarp();
            if (lane == 0) mbar_arrive(&k_empty[ks]);
            tc::fence_after();
            // pass 1: row maximum of the raw scores, 64 columns at a time; a
            // tile with any key outside this row's range takes the masked path
            const bool full = mask == 0xffu && tbase >= qlo && tbase + kKeys - 1 <= qpos && valid_row;
            // key column e of chunk c is attended iff e - lo_c is in [0, hi_c - lo_c]
            // and its block was loaded
            auto mask_chunk = [&](int c, float (&v)[32]) {
                const int32_t lo_c = qlo - (tbase + 32 * c);
                const uint32_t span = static_cast<uint32_t>(qpos - qlo);  // qlo <= qpos
                const uint32_t bm = valid_row ? (mask >> (2 * c)) & 3u : 0u;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const bool ok = static_cast<uint32_t>(e - lo_c) <= span && ((bm >> (e >> 4)) & 1u);
                    v[e] = ok ? v[e] : -INFINITY;
                }
            };
            float mt = -INFINITY;
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {
                float v0[32], v1[32];
                {
                    uint32_t r0[32], r1[32];
                    tc::ld32(sx + 64 * c2, r0);
                    tc::ld32(sx + 64 * c2 + 32, r1);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        v0[e] = __uint_as_float(r0[e]);
                        v1[e] = __uint_as_float(r1[e]);
                    }
                }
                if (!full) {
                    mask_chunk(2 * c2, v0);
                    mask_chunk(2 * c2 + 1, v1);
                }
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = fmaxf(fmaxf(v0[e], v0[8 + e]), fmaxf(v1[e], v1[8 + e]));
#pragma unroll
                for (int c = 2; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        m8[e] = fmaxf(m8[e], fmaxf(v0[8 * c + e], v1[8 * c + e]));
                mt = fmaxf(mt, fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))));
            }
            mt *= sl;
            // keep the reference max within 2^8 of the running max
            const float new_ref = (mt > m_ref + static_cast<float>(kRescaleLog2)) ? mt : m_ref;
            const float alpha = fast_exp2(m_ref - new_ref);  // 0 from -inf, 1 if unchanged
            const bool resc = new_ref != m_ref && m_ref != -INFINITY;
            if (__any_sync(0xffffffffu, resc)) {
                // O_x holds the products up to tile jj-1; S_x(jj) was issued
                // after them, so they are complete
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
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            // pass 2: P = 2^(s * scale - max), 32 columns at a time; group g
            // (16 keys) -> 8 columns of P hi then 8 of P lo, in place
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float v[32];
                {
                    uint32_t r[32];
                    tc::ld32(sx + 32 * c, r);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
                }
                if (!full) mask_chunk(c, v);
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float a = fast_exp2(fmaf(v[16 * g + 2 * e], sl, nmu));
                        const float b = fast_exp2(fmaf(v[16 * g + 2 * e + 1], sl, nmu));
                        ls[e & 3] += a + b;
                        const uint32_t hi = pack_bf16x2(a, b);
                        pk[e] = hi;
                        pk[8 + e] = pack_bf16x2(a - bf16lo_to_f32(hi), b - bf16hi_to_f32(hi));
                    }
                    tc::st16(sx + 32 * c + 16 * g, pk);
                }
            }
            l = l * (resc ? alpha : 1.f) + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
            // value rows of keys outside [kv_lo, kv_hi) or of blocks not
            // loaded hold stale slots (possibly NaN): tile A's warpgroup zeroes
            // them before either P.V product reads them
            const bool edge = mask != 0xffu || tbase < w.kv_lo || tbase + kKeys > w.kv_hi;
            if (x == 0 && edge) {
                const bool landed = mbar_wait(&v_full[ks], (jj >> 1) & 1);
                if (__any_sync(0xffffffffu, !landed)) {
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                    abort = true;
                    break;
                }
                const int kr = row;  // key row of this thread
                const int32_t kp = tbase + kr;
                if (!(kp >= w.kv_lo && kp < w.kv_hi && ((mask >> (kr >> 4)) & 1u))) {
                    uint8_t *vs = v_s + ks * kTileBytes + kr * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        *reinterpret_cast<uint4 *>(vs + c * 16) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(vs + kKVRegion + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
            }
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
        }
        // epilogue: O / l once the tile's last P.V product is in
        if (!abort) {
            const bool done = mbar_wait(&pv_done[x], (ntile - 1) & 1);
            if (__any_sync(0xffffffffu, !done)) {
                if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
            } else {
                tc::fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
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
// host side
// ---------------------------------------------------------------------------
bool prefill_shape_built(pkv_dtype dtype, int32_t D, int32_t bs, int32_t G)
{
    if (G < 1 || G > 16) return false;
    if (dtype == PKV_BF16) return D == pf::kD && bs == 16 && (pf::kRows % G) == 0;
    return (D == 32 || D == 64 || D == 128 || D == 256) && bs <= 64 && bs * D <= 4096 &&
           (kPf32Pairs % G) == 0;
}

int32_t prefill_queries_per_cta(pkv_dtype dtype, int32_t G)
{
    return dtype == PKV_BF16 ? pf::kQTiles * (pf::kRows / G) : kPf32Pairs / G;
}

cudaError_t launch_prefill_bf16(const PrefillParams &p, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, cudaStream_t stream)
{
    const int64_t ctas = static_cast<int64_t>(p.batch) * p.hkv * p.q_tiles;
    if (ctas == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(prefill_bf16_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           pf::kLaunchBytes);
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_PREFILL, stream);
    err = launch_pdl(prefill_bf16_kernel, dim3(static_cast<unsigned>(ctas)), dim3(pf::kThreads),
                     pf::kLaunchBytes, stream, kmap, vmap, p);
    prof_end(PKV_KERNEL_PREFILL, stream);
    return err;
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
