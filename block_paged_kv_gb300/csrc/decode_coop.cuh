// Split-KV paged decode for a few long rows, bf16 pools: the four compute
// warps of a CTA work on every block of the run together, each on a quarter
// of the head dimension ("perf.md": above some context length the pages switch
// decode to grouped, partitioned kernels; this is the layout of such a kernel
// for a grid of about two CTAs per SM).
//
// Why a second layout.  When rows x kv heads are fewer than the SMs, each CTA
// streams one long run of blocks.  If each warp took every fourth block (the
// many-row kernel in decode_kernel.cuh), a warp would keep at most its own
// ring share in flight (one 16 KB block at head_dim 256) and the warps of a
// CTA would drift apart, the CTA then waiting for its slowest one.  Here a
// fifth warp keeps one shared ring of kStages blocks (96 KB) full: it refills
// a stage as soon as the four compute warps have released it, so the ring's
// other blocks stay in flight while two are computed, and every compute warp
// finishes with the last block.
//
// Per pass (two blocks, 32 tokens), compute warp w:
//   S^T partial = K[:, dims of w] Q^T[dims of w, :]   (mma.sync m16n8k16, fp32)
//   the four partials meet in shared memory (one named barrier, which also
//   votes on whether any warp's wait for the blocks ran out), every warp adds
//   them in the same order, so all hold the same scores and the same online
//   softmax state;
//   O^T[dims of w, :] += V^T[dims of w, :] P^T        (P as bf16 hi + lo)
// At the end each warp writes its dims of the partial (unnormalised O, the
// running max in log2 units and the weight sum) to the workspace; the merge
// kernel is the one of the other decode kernels.
#pragma once

#include "decode_kernel.cuh"

namespace pkv {

template <int D>
struct CoopCfg {
    static constexpr int kTok = 16;
    static constexpr int kTileBytes = kTok * D * 2;         // one (block, kv head) tile of K or V
    static constexpr int kStageBytes = 2 * kTileBytes;      // K + V of one block
    static constexpr int kRingBytes = 96 * 1024;
    static constexpr int kStages = kRingBytes / kStageBytes;
    static constexpr int kBpp = 2;                          // blocks per pass
    static constexpr int kKS = D / 16 / kDecodeWarps;       // 16-dim k-steps of a warp's S part
    static constexpr int kMT = D / 16 / kDecodeWarps;       // 16-dim m-tiles of a warp's O part
    static constexpr int kThreads = (kDecodeWarps + 1) * 32;  // + the producer warp
    static constexpr int kSbufOff = kRingBytes;             // [2][warps][kBpp][32 lanes] float4
    static constexpr int kSbufBytes = 2 * kDecodeWarps * kBpp * 32 * 16;
    static constexpr int kBarOff = kSbufOff + kSbufBytes;   // full[kStages], empty[kStages]
    static constexpr int kOkOff = kBarOff + 2 * kStages * 8;  // [kStages] int32: block loaded
    static constexpr int kBytes = kOkOff + kStages * 4;
    static constexpr int kLaunchBytes = kBytes + 1024;      // room to align the base to 1024
    static constexpr int kCtasPerSm = 2;
    static_assert(kStages >= 2 * kBpp, "a pass's blocks plus the next pass's in flight");
    static_assert(kKS >= 1 && D % (16 * kDecodeWarps) == 0, "head_dim splits into four warps");
    static_assert(kCtasPerSm * kLaunchBytes <= 227 * 1024, "two CTAs per SM");
};

// Named barrier 1 over the CTA's compute warps; returns whether any thread
// passed `pred`.
__device__ __forceinline__ bool coop_barrier_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(kDecodeWarps * 32)
        : "memory");
    return r != 0;
}

template <int D>
__device__ __forceinline__ void decode_coop_body(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                                 const DecodeParams &p, const int64_t cta)
{
    using C = CoopCfg<D>;
    constexpr int S = C::kStages;
    constexpr int BPP = C::kBpp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float4 *sbuf = reinterpret_cast<float4 *>(smem + C::kSbufOff);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + S;
    int32_t *stage_ok = reinterpret_cast<int32_t *>(smem + C::kOkOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool producer = warp == kDecodeWarps;
    const int G = p.group;
    const int bs = C::kTok;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    pdl_wait();     // inputs may come from the previous kernel on the stream
    pdl_trigger();  // the merge kernel may be scheduled now; it waits for us

    // ---------------------------------------------------------------- work item
    int64_t bid = cta;
    const int32_t s = static_cast<int32_t>(bid % p.plan.n_suffix_splits);
    bid /= p.plan.n_suffix_splits;
    const int32_t g = static_cast<int32_t>(bid % p.hkv);
    const int32_t r = static_cast<int32_t>(bid / p.hkv);
    const int32_t *table_row = p.tables + static_cast<int64_t>(r) * p.width;
    // the producer fetches the run's block ids before the row's length is
    // known, on the guess that the row's splits start at block 0 (full
    // attention); the compute warps load their query fragments meanwhile
    BlockIds ids;
    const int32_t b_guess = s * p.plan.split_blocks;
    if (producer)
        ids.init(table_row + min(b_guess, p.width), 0, 1,
                 max(0, min(p.plan.split_blocks, p.width - b_guess)), lane);
    // B fragments of Q^T: the G heads of (r, g) on N (one n-tile), this
    // warp's k-steps kk = w * kKS + i on K
    uint32_t qb[C::kKS][2];
    if (!producer) {
        const int row = lane >> 2;
        const bool live = row < G;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(p.q) +
                              (static_cast<int64_t>(r) * p.hq + g * G + (live ? row : 0)) * (D / 2) +
                              (lane & 3);
#pragma unroll
        for (int i = 0; i < C::kKS; ++i) {
            const int kk = warp * C::kKS + i;
            qb[i][0] = live ? __ldg(src + 8 * kk) : 0u;
            qb[i][1] = live ? __ldg(src + 8 * kk + 4) : 0u;
        }
    }
    const RowRange rr = row_range(p, r, s == 0 && g == 0);
    const int32_t b0 = rr.b_first + s * p.plan.split_blocks;
    const int32_t b1 = min(b0 + p.plan.split_blocks, rr.b_end);
    if (b0 >= b1) return;  // uniform over the CTA
    const int32_t nblk = b1 - b0;
    const int32_t lo_all = rr.lo, hi_all = rr.L;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kDecodeWarps);  // lane 0 of every compute warp
        }
        fence_mbar_init();
    }
    __syncthreads();

    auto withheld = [&](int32_t j) { return (p.drill & kDrillWithholdFirst) != 0 && j == 0; };
    if (producer) {
        // ------------------------------------------------------------- loads
        // block j of the run goes to stage j % S once the compute warps have
        // released block j - S
        if (rr.b_first != 0)
            ids.init(table_row + b0, 0, 1, nblk, lane);  // the guess was wrong
        else
            ids.n = nblk;  // fetched ids past the run are never used
        const uint64_t policy = l2_evict_first_policy();
        int32_t j = 0;
        for (; j < nblk; ++j) {
            const int st = j % S;
            if (j >= S) {
                bool freed = true;
                if (lane == 0) freed = mbar_wait(&empty[st], ((j / S) - 1) & 1, p.wait_ns);
                if (!__shfl_sync(0xffffffffu, freed, 0)) {
                    if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
                    break;
                }
            }
            const int32_t id = ids.next(j, lane);
            if (lane == 0 && !withheld(j)) {
                const bool ok = static_cast<uint32_t>(id) < static_cast<uint32_t>(p.num_blocks);
                stage_ok[st] = ok ? 1 : 0;  // published by the arrive (release)
                if (ok) {
                    mbar_arrive_expect_tx(&full[st], 2 * C::kTileBytes);
                    uint8_t *kdst = smem + st * C::kStageBytes;
                    tma_load_5d(kdst, &kmap, &full[st], 0, 0, 0, g, id, policy);
                    tma_load_5d(kdst + C::kTileBytes, &vmap, &full[st], 0, 0, 0, g, id, policy);
                } else {
                    report(p.status, PKV_DEV_BAD_BLOCK);
                    mbar_arrive(&full[st]);  // an empty stage: tokens masked, values unread
                }
            }
        }
        // every copy this warp issued has landed before it leaves (at a
        // normal end the compute warps wait for them anyway; after a wait
        // ran out they may have left already)
        if (lane == 0)
            for (int32_t t = max(0, j - S); t < j; ++t)
                if (!withheld(t)) mbar_wait(&full[t % S], (t / S) & 1);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- compute
    const int g8 = lane >> 2;  // C rows g8, g8 + 8 (tokens / dims); B column g8
    const int cc = lane & 3;   // C columns 2cc, 2cc + 1 (query rows)
    const int ka_tok = ((lane >> 3) & 1) * 8 + (lane & 7), ka_dof = (lane >> 4) * 8;
    const int va_tok = (lane >> 4) * 8 + (lane & 7), va_dof = ((lane >> 3) & 1) * 8;
    float oT[C::kMT][4];
#pragma unroll
    for (int i = 0; i < C::kMT; ++i) oT[i][0] = oT[i][1] = oT[i][2] = oT[i][3] = 0.f;
    float mc[2] = {-INFINITY, -INFINITY}, lc[2] = {0.f, 0.f};
    const int32_t npass = (nblk + BPP - 1) / BPP;
    for (int32_t k = 0; k < npass; ++k) {
        bool got = true, okb[BPP], have[BPP];
        uint32_t kt[BPP];
        int bt[BPP];
#pragma unroll
        for (int b = 0; b < BPP; ++b) {
            const int32_t j = k * BPP + b;
            const int st = j % S;
            have[b] = j < nblk;
            if (have[b]) got = got && mbar_wait(&full[st], (j / S) & 1, p.wait_ns);
            okb[b] = have[b] && got && stage_ok[st] != 0;
            kt[b] = smem_u32(smem + st * C::kStageBytes);
            bt[b] = (b0 + j) * bs;
        }
        // this warp's part of S^T = K Q^T for each block: tokens on M, the G
        // heads on N
        float sa[BPP][4];
#pragma unroll
        for (int b = 0; b < BPP; ++b) {
            sa[b][0] = sa[b][1] = sa[b][2] = sa[b][3] = 0.f;
            if (okb[b]) {
#pragma unroll
                for (int i = 0; i < C::kKS; ++i) {
                    uint32_t a[4];
                    ldsm_x4(kv_chunk_addr(kt[b], ka_tok, (warp * C::kKS + i) * 16 + ka_dof), a[0], a[1],
                            a[2], a[3]);
                    mma_16816(sa[b], a, qb[i][0], qb[i][1]);
                }
            }
        }
        float4 *slot = sbuf + (k & 1) * (kDecodeWarps * BPP * 32);
#pragma unroll
        for (int b = 0; b < BPP; ++b)
            slot[(warp * BPP + b) * 32 + lane] = make_float4(sa[b][0], sa[b][1], sa[b][2], sa[b][3]);
        if (coop_barrier_any(!got)) {
            // a wait ran out (every compute warp sees it here); the producer
            // lets its copies land before it leaves
            if (lane == 0) report(p.status, PKV_DEV_TIMEOUT);
            return;
        }
        // the whole S^T of each block, mask, scale to log2 units; element e:
        // token g8 + 8(e/2), column 2cc + e%2
        float sv[BPP][4];
#pragma unroll
        for (int b = 0; b < BPP; ++b) {
            float sT[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const float4 v = slot[(w * BPP + b) * 32 + lane];
                sT[0] += v.x;
                sT[1] += v.y;
                sT[2] += v.z;
                sT[3] += v.w;
            }
            if (okb[b] && bt[b] >= lo_all && bt[b] + bs <= hi_all) {
#pragma unroll
                for (int e = 0; e < 4; ++e) sv[b][e] = sT[e] * p.scale_log2;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = bt[b] + g8 + 8 * (e >> 1);
                    sv[b][e] = (okb[b] && pos >= lo_all && pos < hi_all) ? sT[e] * p.scale_log2 : -INFINITY;
                }
            }
        }
        // column maxima over the pass's tokens: this lane's, then the 8 lanes of cc
        float mu[2], al[2];
        bool grew = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float mx = -INFINITY;
#pragma unroll
            for (int b = 0; b < BPP; ++b) mx = fmaxf(mx, fmaxf(sv[b][e], sv[b][e + 2]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(mc[e], mx);
            mu[e] = mn == -INFINITY ? 0.f : mn;
            al[e] = fast_exp2(mc[e] - mu[e]);
            grew = grew || mn != mc[e];
            mc[e] = mn;
        }
        float pv[BPP][4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float sum = 0.f;
#pragma unroll
            for (int b = 0; b < BPP; ++b) {
                pv[b][e] = fast_exp2(sv[b][e] - mu[e]);
                pv[b][e + 2] = fast_exp2(sv[b][e + 2] - mu[e]);
                sum += pv[b][e] + pv[b][e + 2];
            }
            lc[e] = lc[e] * al[e] + sum;
        }
        if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
            for (int i = 0; i < C::kMT; ++i) {
                oT[i][0] *= al[0];
                oT[i][1] *= al[1];
                oT[i][2] *= al[0];
                oT[i][3] *= al[1];
            }
        }
        // O^T += V^T P^T per block: P as a bf16 pair hi + lo (B fragment
        // through movmatrix.trans), values of tokens outside the range zeroed
        // (stale slots may hold NaN)
#pragma unroll
        for (int b = 0; b < BPP; ++b) {
            if (!okb[b]) continue;
            const uint32_t vt = kt[b] + C::kTileBytes;
            const uint32_t h0 = pack_bf16x2(pv[b][0], pv[b][1]);
            const uint32_t h1 = pack_bf16x2(pv[b][2], pv[b][3]);
            const uint32_t l0 = pack_bf16x2(pv[b][0] - bf16lo_to_f32(h0), pv[b][1] - bf16hi_to_f32(h0));
            const uint32_t l1 = pack_bf16x2(pv[b][2] - bf16lo_to_f32(h1), pv[b][3] - bf16hi_to_f32(h1));
            const uint32_t pb0 = movmatrix_trans(h0), pb1 = movmatrix_trans(h1);
            const uint32_t pl0 = movmatrix_trans(l0), pl1 = movmatrix_trans(l1);
            uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
            if (bt[b] < lo_all || bt[b] + bs > hi_all) {
                const int t0 = bt[b];
                auto live = [&](int t) { return t0 + t >= lo_all && t0 + t < hi_all; };
                mk0 = (live(2 * cc) ? 0x0000ffffu : 0u) | (live(2 * cc + 1) ? 0xffff0000u : 0u);
                mk1 = (live(2 * cc + 8) ? 0x0000ffffu : 0u) | (live(2 * cc + 9) ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int i = 0; i < C::kMT; ++i) {
                uint32_t a[4];
                ldsm_x4_trans(kv_chunk_addr(vt, va_tok, (warp * C::kMT + i) * 16 + va_dof), a[0], a[1],
                              a[2], a[3]);
                a[0] &= mk0;
                a[1] &= mk0;
                a[2] &= mk1;
                a[3] &= mk1;
                mma_16816(oT[i], a, pb0, pb1);
                mma_16816(oT[i], a, pl0, pl1);
            }
        }
        // release the pass's stages: these generic-proxy reads come before
        // the producer's async-proxy refill
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
#pragma unroll
            for (int b = 0; b < BPP; ++b)
                if (have[b]) mbar_arrive(&empty[(k * BPP + b) % S]);
    }

    // column sums over the 8 lanes sharing cc
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        lc[e] += __shfl_xor_sync(0xffffffffu, lc[e], 4);
        lc[e] += __shfl_xor_sync(0xffffffffu, lc[e], 8);
        lc[e] += __shfl_xor_sync(0xffffffffu, lc[e], 16);
    }
    // element e of oT[i]: dim 16(w kMT + i) + g8 + 8(e/2), query row 2cc + e%2
    const int32_t slot = p.plan.n_prefix_splits + s;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int row = 2 * cc + e;
        if (row >= G) continue;
        const size_t pi = partial_index(p, r, g * G + row, slot);
        float *dst = p.ws_o + pi * D + warp * C::kMT * 16 + g8;
#pragma unroll
        for (int i = 0; i < C::kMT; ++i) {
            dst[16 * i] = oT[i][e];
            dst[16 * i + 8] = oT[i][e + 2];
        }
        if (warp == 0 && g8 == 0)
            *reinterpret_cast<float2 *>(p.ws_ml + pi * 2) = make_float2(mc[e], lc[e]);
    }
}

template <int D>
__global__ void __launch_bounds__(CoopCfg<D>::kThreads, CoopCfg<D>::kCtasPerSm)
    decode_coop_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const DecodeParams p)
{
    decode_coop_body<D>(kmap, vmap, p, blockIdx.x);
}

template <int D>
__global__ void __launch_bounds__(CoopCfg<D>::kThreads, CoopCfg<D>::kCtasPerSm)
    decode_coop_grouped_kernel(const __grid_constant__ GroupedDecode gd)
{
    int i = 0;
    const int64_t b = blockIdx.x;
    while (i + 1 < gd.n && b >= gd.cta_end[i]) ++i;
    const int64_t first = i > 0 ? gd.cta_end[i - 1] : 0;
    decode_coop_body<D>(gd.kmap[i], gd.vmap[i], gd.g[i], b - first);
}

template <int D>
static cudaError_t launch_coop(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, cudaStream_t stream)
{
    const int64_t ctas = p.plan.n_suffix_ctas;
    if (ctas == 0) return cudaSuccess;
    auto kern = decode_coop_kernel<D>;
    const int smem = CoopCfg<D>::kLaunchBytes;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_DECODE_SPLIT, stream);
    err = launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(CoopCfg<D>::kThreads), smem,
                     stream, kmap, vmap, p);
    prof_end(PKV_KERNEL_DECODE_SPLIT, stream);
    return err;
}

template <int D>
static cudaError_t launch_coop_grouped(const GroupedDecode &gd, cudaStream_t stream)
{
    const int64_t ctas = gd.cta_end[gd.n - 1];
    if (ctas == 0) return cudaSuccess;
    auto kern = decode_coop_grouped_kernel<D>;
    const int smem = CoopCfg<D>::kLaunchBytes;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    prof_begin(PKV_KERNEL_DECODE_SPLIT, stream);
    err = launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(CoopCfg<D>::kThreads), smem, stream,
                     gd);
    prof_end(PKV_KERNEL_DECODE_SPLIT, stream);
    return err;
}

}  // namespace pkv
