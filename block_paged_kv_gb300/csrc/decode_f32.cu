// Split-KV paged decode for f32 pools (CUDA cores) and the log-sum-exp merge
// of split partials used by every decode path ("perf.md", partition-rule
// paragraphs: each partition keeps online-softmax partials that a reducer
// merges; an empty partition contributes exact zeros).
//
// The f32 kernel follows the same work items and partial layout as the bf16
// kernel: a CTA takes up to 16 (row, q head) pairs of one kv head (the G heads
// of a row, or pairs of a shared-prefix group) and a run of blocks; each block
// tile is staged in shared memory and scores, softmax and values are
// accumulated in fp32.
#include "decode_common.cuh"

namespace pkv {

constexpr int kF32Threads = 128;

__global__ void __launch_bounds__(kF32Threads)
    decode_f32_kernel(const DecodeParams p, int prefix_mode)
{
    constexpr int NQ = kF32Rows;
    extern __shared__ float fsm[];
    const int D = p.head_dim, bs = p.block_size;
    float *qs = fsm;                   // [NQ][D]
    float *os = qs + NQ * D;           // [NQ][D]
    float *ks = os + NQ * D;           // [bs][D]
    float *vs = ks + bs * D;           // [bs][D]
    float *sc = vs + bs * D;           // [NQ][bs]
    float *mrow = sc + NQ * bs;        // [NQ]
    float *lrow = mrow + NQ;           // [NQ]
    float *alpha = lrow + NQ;          // [NQ]
    int32_t *prow = reinterpret_cast<int32_t *>(alpha + NQ);  // [NQ] row, -1 = unused
    int32_t *phead = prow + NQ;        // [NQ]
    int32_t *plo = phead + NQ;         // [NQ]
    int32_t *phi = plo + NQ;           // [NQ]
    int32_t *misc = phi + NQ;          // [0] = table row

    const int tid = threadIdx.x;
    const int G = p.group;
    pdl_wait();
    pdl_trigger();
    int32_t b0, nblk, slot, g;
    if (!prefix_mode) {
        int64_t bid = blockIdx.x;
        const int32_t s = static_cast<int32_t>(bid % p.plan.n_suffix_splits);
        bid /= p.plan.n_suffix_splits;
        g = static_cast<int32_t>(bid % p.hkv);
        const int32_t r = static_cast<int32_t>(bid / p.hkv);
        const RowRange rr = row_range(p, r, s == 0 && g == 0);
        b0 = rr.b_first + s * p.plan.split_blocks;
        const int32_t b1 = min(b0 + p.plan.split_blocks, rr.b_end);
        if (b0 >= b1) return;
        nblk = b1 - b0;
        slot = p.plan.n_prefix_splits + s;
        if (tid < NQ) {
            prow[tid] = tid < G ? r : -1;
            phead[tid] = g * G + tid;
            plo[tid] = rr.lo;
            phi[tid] = rr.L;
        }
        if (tid == 0) misc[0] = r;
    } else {
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
        if (tid < NQ) prow[tid] = -1;
        __syncthreads();
        if (tid < 32) {
            const int lane = tid;
            int32_t cnt = 0, leader = -1;
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
                    if ((rank + 1) * G > p.plan.prefix_chunks * NQ)
                        report(p.status, PKV_DEV_BAD_PREFIX);  // more rows than max_group_rows
                    for (int j = 0; j < G; ++j) {
                        const int32_t k = rank * G + j - chunk * NQ;
                        if (k >= 0 && k < NQ) {
                            prow[k] = r;
                            phead[k] = g * G + j;
                            plo[k] = 0;
                            phi[k] = L;
                        }
                    }
                }
                cnt += __popc(m);
            }
            leader = __reduce_max_sync(0xffffffffu, leader);
            if (lane == 0) misc[0] = leader;
        }
    }
    __syncthreads();
    if (prow[0] < 0) return;
    const int32_t tab_row = misc[0];
    if (prefix_mode) {
        for (int i = tid; i < NQ * nblk; i += kF32Threads) {
            const int k = i / nblk, b = b0 + i % nblk;
            const int32_t pr = prow[k];
            if (pr >= 0 && (k % G) == 0 &&
                __ldg(p.tables + static_cast<int64_t>(pr) * p.width + b) !=
                    __ldg(p.tables + static_cast<int64_t>(tab_row) * p.width + b))
                report(p.status, PKV_DEV_BAD_PREFIX);
        }
    }
    const float *qg = static_cast<const float *>(p.q);
    for (int i = tid; i < NQ * D; i += kF32Threads) {
        const int k = i / D, d = i % D;
        qs[i] = prow[k] >= 0 ? qg[(static_cast<int64_t>(prow[k]) * p.hq + phead[k]) * D + d] : 0.f;
        os[i] = 0.f;
    }
    if (tid < NQ) {
        mrow[tid] = -INFINITY;
        lrow[tid] = 0.f;
    }
    __syncthreads();

    const float *kpool = static_cast<const float *>(p.k_pool);
    const float *vpool = static_cast<const float *>(p.v_pool);
    for (int i = 0; i < nblk; ++i) {
        const int32_t b = b0 + i;
        const int32_t blk = __ldg(p.tables + static_cast<int64_t>(tab_row) * p.width + b);
        const bool ok = static_cast<uint32_t>(blk) < static_cast<uint32_t>(p.num_blocks);
        if (!ok && tid == 0) report(p.status, PKV_DEV_BAD_BLOCK);
        if (ok) {
            const int64_t base = (static_cast<int64_t>(blk) * p.hkv + g) * bs * D;
            for (int j = tid; j < bs * D; j += kF32Threads) {
                ks[j] = __ldg(kpool + base + j);
                vs[j] = __ldg(vpool + base + j);
            }
        }
        __syncthreads();
        for (int j = tid; j < NQ * bs; j += kF32Threads) {
            const int k = j / bs, t = j % bs;
            const int pos = b * bs + t;
            float sv = -INFINITY;
            if (ok && prow[k] >= 0 && pos >= plo[k] && pos < phi[k]) {
                float acc = 0.f;
                for (int d = 0; d < D; ++d) acc = fmaf(qs[k * D + d], ks[t * D + d], acc);
                sv = acc * p.scale_log2;
            }
            sc[j] = sv;
        }
        __syncthreads();
        if (tid < NQ) {
            float mx = -INFINITY;
            for (int t = 0; t < bs; ++t) mx = fmaxf(mx, sc[tid * bs + t]);
            const float mn = fmaxf(mrow[tid], mx);
            const float mu = mn == -INFINITY ? 0.f : mn;
            const float al = fast_exp2(mrow[tid] - mu);
            float sum = 0.f;
            for (int t = 0; t < bs; ++t) {
                const float e = fast_exp2(sc[tid * bs + t] - mu);
                sc[tid * bs + t] = e;
                sum += e;
            }
            lrow[tid] = lrow[tid] * al + sum;
            mrow[tid] = mn;
            alpha[tid] = al;
        }
        __syncthreads();
        for (int j = tid; j < NQ * D; j += kF32Threads) {
            const int k = j / D, d = j % D;
            float acc = os[j] * alpha[k];
            for (int t = 0; t < bs; ++t) {
                const float w = sc[k * bs + t];
                if (w != 0.f) acc = fmaf(w, vs[t * D + d], acc);  // masked slots may hold NaN
            }
            os[j] = acc;
        }
        __syncthreads();
    }
    for (int j = tid; j < NQ * D; j += kF32Threads) {
        const int k = j / D, d = j % D;
        if (prow[k] < 0) continue;
        const size_t pi = partial_index(p, prow[k], phead[k], slot);
        p.ws_o[pi * D + d] = os[j];
        if (d == 0) {
            p.ws_ml[pi * 2] = mrow[k];
            p.ws_ml[pi * 2 + 1] = lrow[k];
        }
    }
}

size_t f32_smem_bytes(int D, int bs)
{
    return sizeof(float) * (2 * kF32Rows * D + 2 * bs * D + kF32Rows * bs + 3 * kF32Rows) +
           sizeof(int32_t) * (4 * kF32Rows + 4);
}

cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t stream)
{
    const size_t smem = f32_smem_bytes(p.head_dim, p.block_size);
    cudaError_t err = cudaFuncSetAttribute(decode_f32_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    if (p.plan.n_prefix_ctas > 0) {
        prof_begin(PKV_KERNEL_DECODE_PREFIX, stream);
        err = launch_pdl(decode_f32_kernel, dim3(static_cast<unsigned>(p.plan.n_prefix_ctas)),
                         dim3(kF32Threads), smem, stream, p, 1);
        prof_end(PKV_KERNEL_DECODE_PREFIX, stream);
        if (err != cudaSuccess) return err;
    }
    if (p.plan.n_suffix_ctas > 0) {
        prof_begin(PKV_KERNEL_DECODE_SPLIT, stream);
        err = launch_pdl(decode_f32_kernel, dim3(static_cast<unsigned>(p.plan.n_suffix_ctas)),
                         dim3(kF32Threads), smem, stream, p, 0);
        prof_end(PKV_KERNEL_DECODE_SPLIT, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Merge of the split partials.  With W = 1 (rows with few partials) an item is
// a (row, q head) and a warp takes it whole; with W = 8 an item is a (row,
// q head, chunk of up to 64 dims) shared by the CTA's 8 warps: warp w takes partials w, w+W, ...  M = max of the
// partial maxima; each partial is weighted by 2^(m_s - M); out = sum w_s O_s /
// sum w_s l_s.  Each warp first reduces its own partials against its own
// maximum and the warp results are merged through shared memory, so a row with
// many partials keeps many loads in flight.  Rows with no partial (an empty
// key range) get zeros.
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ OutT to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

constexpr int kCombineWarps = 8;

template <typename OutT, int D, int W, int KB>
__device__ __forceinline__ void decode_combine_body(const DecodeParams &p, const int64_t cta)
{
    constexpr int CH = (W == 1 || D < 64) ? D : 64;  // dims per item
    constexpr int PER = CH / 32;                     // dims per lane
    constexpr int NCH = D / CH;
    constexpr int IPC = kCombineWarps / W;  // items per CTA
    __shared__ float sm_m[kCombineWarps], sm_l[kCombineWarps];
    __shared__ float sm_acc[kCombineWarps][CH];
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warp = wid % W, sub = wid / W;  // warp within the item, item within the CTA
    const int64_t item = cta * IPC + sub;
    bool live = item < static_cast<int64_t>(p.batch) * p.max_q * p.hq * NCH;
    const int64_t idx = live ? item / NCH : 0;  // ((row, query), q head)
    const int ch = static_cast<int>(item % NCH);
    // The row bookkeeping reads only call inputs: the decode kernel released
    // this grid after its own wait on earlier work, so they are final already.
    const int32_t h = static_cast<int32_t>(idx % p.hq);
    const int32_t r = static_cast<int32_t>(idx / p.hq / p.max_q);
    const int32_t t = static_cast<int32_t>((idx / p.hq) % p.max_q);
    const RowRange rr = row_range(p, r, false);
    live = live && t < rr.C;  // a row with fewer queries than max_q
    const int32_t npre = row_prefix_splits(p, rr);
    const int32_t n = live ? npre + row_suffix_splits(p, rr) : 0;
    const int64_t out_row = static_cast<int64_t>(rr.q0) + t;  // packed query index
    pdl_wait();  // the partials come from the decode kernel just before
    const size_t base = partial_index(p, r, h, 0, t);
    auto slot_of = [&](int32_t k) { return k < npre ? k : p.plan.n_prefix_splits + (k - npre); };

    // this warp's partials k = warp + W * i, in batches of kB: every load of
    // a batch is issued before any of them is used (one memory round trip per
    // batch), and each batch is folded into the running (max, sum, values)
    // with the usual rescale (a factor of exactly 0 while nothing has been
    // seen).  The launch sizes KB to the row's partials, so that one batch
    // usually covers them, without more registers (fewer resident CTAs) than
    // that needs.
    constexpr int kB = (W == 1 && PER > 4) ? KB / 2 : KB;
    float Mw = -INFINITY, lw = 0.f;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int32_t k0 = warp; k0 < n; k0 += W * kB) {
        float2 ml[kB];
        float v[kB][PER];
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            const int32_t k = k0 + W * i;
            if (k < n) {
                const size_t slot = base + slot_of(k);
                ml[i] = *reinterpret_cast<const float2 *>(p.ws_ml + slot * 2);
                const float *src = p.ws_o + slot * D + ch * CH + (W == 1 ? lane : lane * PER);
                if constexpr (W == 1) {
                    // lane owns dims lane + 32 e: each load instruction is coalesced
#pragma unroll
                    for (int e = 0; e < PER; ++e) v[i][e] = src[32 * e];
                } else if constexpr (PER == 2) {
                    const float2 t = *reinterpret_cast<const float2 *>(src);
                    v[i][0] = t.x;
                    v[i][1] = t.y;
                } else {
                    v[i][0] = src[0];
                }
            } else {
                ml[i] = make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int e = 0; e < PER; ++e) v[i][e] = 0.f;
            }
        }
        float bm = Mw;
#pragma unroll
        for (int i = 0; i < kB; ++i) bm = fmaxf(bm, ml[i].x);
        if (bm != -INFINITY) {
            const float a = fast_exp2(Mw - bm);
            lw *= a;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] *= a;
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const float wgt = fast_exp2(ml[i].x - bm);  // 0 for an empty partial
                lw = fmaf(wgt, ml[i].y, lw);
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] = fmaf(wgt, v[i][e], acc[e]);
            }
            Mw = bm;
        }
    }
    if constexpr (W == 1) {
        // one warp per item: every lane already holds the item's sum
        if (!live) return;
        const float inv = lw > 0.f ? 1.f / lw : 0.f;
        OutT *out = static_cast<OutT *>(p.out) + (out_row * p.hq + h) * D + lane;
#pragma unroll
        for (int e = 0; e < PER; ++e) out[32 * e] = to_out<OutT>(acc[e] * inv);
    } else {
        if (lane == 0) {
            sm_m[wid] = Mw;
            sm_l[wid] = lw;
        }
#pragma unroll
        for (int e = 0; e < PER; ++e) sm_acc[wid][lane * PER + e] = acc[e];
        __syncthreads();
        if (live && threadIdx.x < CH) {
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < W; ++i) M = fmaxf(M, sm_m[i]);
            float L = 0.f, o = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int i = 0; i < W; ++i) {
                    const float f = fast_exp2(sm_m[i] - M);  // 0 for a warp without partials
                    L = fmaf(f, sm_l[i], L);
                    o = fmaf(f, sm_acc[i][threadIdx.x], o);
                }
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            static_cast<OutT *>(p.out)[(out_row * p.hq + h) * D + ch * CH + threadIdx.x] = to_out<OutT>(o * inv);
        }
    }
}

template <typename OutT, int D, int W, int KB>
__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const DecodeParams p)
{
    decode_combine_body<OutT, D, W, KB>(p, blockIdx.x);
}

// The merges of several decode calls in one launch: CTAs
// [item_end[i-1], item_end[i]) merge group i.
template <typename OutT, int D, int W, int KB>
__global__ void __launch_bounds__(kCombineWarps * 32)
    decode_combine_grouped_kernel(const __grid_constant__ GroupedDecode gd)
{
    int i = 0;
    const int64_t b = blockIdx.x;
    while (i + 1 < gd.n && b >= gd.item_end[i]) ++i;
    const int64_t first = i > 0 ? gd.item_end[i - 1] : 0;
    decode_combine_body<OutT, D, W, KB>(gd.g[i], b - first);
}

// merge CTAs of one call
template <int W>
static int64_t combine_ctas(const DecodeParams &p)
{
    const int64_t chunks = (W == 1 || p.head_dim < 64) ? 1 : p.head_dim / 64;
    const int64_t items = static_cast<int64_t>(p.batch) * p.max_q * p.hq * chunks;
    const int64_t ipc = kCombineWarps / W;
    return (items + ipc - 1) / ipc;
}

template <typename OutT, int W, int KB>
static cudaError_t launch_combine_grouped_w(GroupedDecode &gd, cudaStream_t stream)
{
    int64_t total = 0;
    for (int i = 0; i < gd.n; ++i) {
        total += combine_ctas<W>(gd.g[i]);
        gd.item_end[i] = total;
    }
    if (total == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(total)), block(kCombineWarps * 32);
    switch (gd.g[0].head_dim) {
    case 64: return launch_pdl(decode_combine_grouped_kernel<OutT, 64, W, KB>, grid, block, 0, stream, gd);
    case 128: return launch_pdl(decode_combine_grouped_kernel<OutT, 128, W, KB>, grid, block, 0, stream, gd);
    case 256: return launch_pdl(decode_combine_grouped_kernel<OutT, 256, W, KB>, grid, block, 0, stream, gd);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_combine_grouped(GroupedDecode &gd, pkv_dtype out_dtype, cudaStream_t stream)
{
    int32_t nslot = 0;  // the shape follows the group with the most partials per row
    for (int i = 0; i < gd.n; ++i) nslot = std::max(nslot, gd.g[i].plan.nslot);
    prof_begin(PKV_KERNEL_DECODE_COMBINE, stream);
    cudaError_t err;
    if (out_dtype == PKV_BF16)
        err = nslot <= 16 ? launch_combine_grouped_w<__nv_bfloat16, 1, 8>(gd, stream)
              : nslot <= 32 ? launch_combine_grouped_w<__nv_bfloat16, kCombineWarps, 4>(gd, stream)
                            : launch_combine_grouped_w<__nv_bfloat16, kCombineWarps, 16>(gd, stream);
    else
        err = nslot <= 16 ? launch_combine_grouped_w<float, 1, 8>(gd, stream)
              : nslot <= 32 ? launch_combine_grouped_w<float, kCombineWarps, 4>(gd, stream)
                            : launch_combine_grouped_w<float, kCombineWarps, 16>(gd, stream);
    prof_end(PKV_KERNEL_DECODE_COMBINE, stream);
    return err;
}

template <typename OutT, int W, int KB>
static cudaError_t launch_combine_w(const DecodeParams &p, cudaStream_t stream)
{
    const int64_t chunks = (W == 1 || p.head_dim < 64) ? 1 : p.head_dim / 64;
    const int64_t items = static_cast<int64_t>(p.batch) * p.max_q * p.hq * chunks;
    const int64_t ipc = kCombineWarps / W;
    const dim3 grid(static_cast<unsigned>((items + ipc - 1) / ipc)), block(kCombineWarps * 32);
    switch (p.head_dim) {
    case 32: return launch_pdl(decode_combine_kernel<OutT, 32, W, KB>, grid, block, 0, stream, p);
    case 64: return launch_pdl(decode_combine_kernel<OutT, 64, W, KB>, grid, block, 0, stream, p);
    case 128: return launch_pdl(decode_combine_kernel<OutT, 128, W, KB>, grid, block, 0, stream, p);
    case 256: return launch_pdl(decode_combine_kernel<OutT, 256, W, KB>, grid, block, 0, stream, p);
    default: return cudaErrorInvalidValue;
    }
}

template <typename OutT>
static cudaError_t launch_combine_t(const DecodeParams &p, cudaStream_t stream)
{
    if (static_cast<int64_t>(p.batch) * p.hq == 0) return cudaSuccess;
    prof_begin(PKV_KERNEL_DECODE_COMBINE, stream);
    // a warp per item while rows have few partials (one batch of 4, or two
    // of 8 at most), eight when they have many: one batch of 4 per warp up to 32
    // partials (few registers, many resident CTAs), else batches of 16
    const int32_t n = p.plan.nslot;
    const cudaError_t err = n <= 4    ? launch_combine_w<OutT, 1, 4>(p, stream)
                            : n <= 16 ? launch_combine_w<OutT, 1, 8>(p, stream)
                            : n <= 32 ? launch_combine_w<OutT, kCombineWarps, 4>(p, stream)
                                      : launch_combine_w<OutT, kCombineWarps, 16>(p, stream);
    prof_end(PKV_KERNEL_DECODE_COMBINE, stream);
    return err;
}

cudaError_t launch_decode_combine(const DecodeParams &p, pkv_dtype dtype, cudaStream_t stream)
{
    return dtype == PKV_BF16 ? launch_combine_t<__nv_bfloat16>(p, stream)
                             : launch_combine_t<float>(p, stream);
}

}  // namespace pkv
