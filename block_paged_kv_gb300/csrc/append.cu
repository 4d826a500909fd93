// Append of new K/V rows into their pool slots ("perf.md", paged knob table:
// the graph-native paged K/V write, MLX_PAGED_NATIVE_KV_WRITE).
//
// One thread moves one 16-byte vector of one (token, kv head) row for both K
// and V: two 16-byte loads and two 16-byte stores, all coalesced within the
// row (a bf16 head_dim-128 row is 16 vectors).  HBM bound: the algorithmic
// traffic is 2 x (read + write) x num_tokens x Hkv x head_dim x elem bytes plus
// 4 bytes of slot per token.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int VPT>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p)
{
    // vector v of row (t, h):  idx = (t * hkv + h) * vecs_per_row + v
    pdl_wait();
    pdl_trigger();
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.hkv * p.vecs_per_row;
    // each block covers VPT * blockDim consecutive vectors, one warp-wide
    // contiguous run per unrolled step
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int64_t idx =
            (static_cast<int64_t>(blockIdx.x) * VPT + u) * blockDim.x + threadIdx.x;
        if (idx >= total) return;
        const int32_t v = static_cast<int32_t>(idx % p.vecs_per_row);
        const int64_t th = idx / p.vecs_per_row;
        const int32_t h = static_cast<int32_t>(th % p.hkv);
        const int32_t t = static_cast<int32_t>(th / p.hkv);
        const int32_t slot = __ldg(p.slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (h == 0 && v == 0) report(p.status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int32_t blk = slot / p.block_size;
        const int32_t off = slot - blk * p.block_size;
        const int64_t dst = ((static_cast<int64_t>(blk) * p.hkv + h) * p.block_size + off) *
                                p.vecs_per_row + v;
        const uint4 kv = __ldcs(reinterpret_cast<const uint4 *>(p.k_new) + idx);
        const uint4 vv = __ldcs(reinterpret_cast<const uint4 *>(p.v_new) + idx);
        reinterpret_cast<uint4 *>(p.k_pool)[dst] = kv;
        reinterpret_cast<uint4 *>(p.v_pool)[dst] = vv;
    }
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.hkv * p.vecs_per_row;
    if (total == 0) return cudaSuccess;
    constexpr int kVpt = 2;
    const int64_t blocks = (total + kVpt * 256 - 1) / (kVpt * 256);
    prof_begin(PKV_KERNEL_APPEND, stream);
    const cudaError_t err = launch_pdl(append_kernel<kVpt>, dim3(static_cast<unsigned>(blocks)),
                                       dim3(256), 0, stream, p);
    prof_end(PKV_KERNEL_APPEND, stream);
    return err;
}

// FP8 append ("perf.md", quantisation scheme table: FP8 KV cache with
// per-layer scales).  Each bf16 element x becomes the E4M3 code of the
// float32 quotient x / scale (correctly rounded; round to nearest even to
// E4M3, saturating), decided without a division (quotient_for_e4m3).
//
// One warp per (token, group of kv heads), head_dim / 4 work items of 4
// codes each per kv head (one 4-byte word of the tile per item).
//   K: a token's codes are 16-byte runs of the tile (4 dims x 4 16-dim
//      steps); item (run, step) quantizes one step's 4 dims.
//   V is stored token-minor: a 4-byte word holds one dim of tokens
//      {2c, 2c+1, 2c+8, 2c+9}.  When the token's block receives all 16 of
//      its tokens in order from this call (tokens t - off .. t - off + 15),
//      the 16 warps of the block share its V words: the warp of offset off
//      writes the words of token quad off / 4 for a quarter of the dims,
//      each from 4 tokens' rows.  Otherwise (a decode step's token, the
//      ragged ends of a chunk) the warp stores its own token's V codes byte
//      by byte.
// E4M3 codes of correctly rounded float32 quotients x / s (s > 0) without a
// division, r = the rounded reciprocal of s.
//
// The product q = x * r lies within 2.5 ulps of the rounded quotient (two
// roundings of at most half an ulp each, and the quotient's own half ulp).
// The code can only differ where the quotient is near a rounding boundary
// of E4M3: a midpoint m between neighbouring E4M3 values, whose float32
// form ends in 19 zero bits.  So unless q is within 4 ulps of such an m it
// is converted as it is.  Near m, the rounded quotient is m itself when
// |x/s - m| <= ulp(m)/2 (a tie goes to m, whose last bit is 0), else one of
// its neighbours; the test is exact: the residual x - s*m is small (a few
// ulps of m, times s) and has at most 9 significant bits, so one fused
// multiply-add yields it exactly (the exact-remainder property used in
// Markstein's division, "Computation of elementary functions on the IBM
// RISC System/6000 processor", 1990), and s * ulp(m)/2 is a power-of-two
// scaling of s.  Zero, NaN, values below 2^-11 (code 0) and above 512
// (saturated to 448) need no test.
__device__ __forceinline__ bool near_e4m3_boundary(float q)
{
    const uint32_t low = __float_as_uint(q) & 0x7FFFFu;
    const float aq = fabsf(q);
    return (low <= 4u || low >= 0x7FFFBu) && aq >= 0x1p-11f && aq <= 512.f;
}

// q = x * r near a boundary: the value to convert in its place
__device__ __forceinline__ float resolve_near_boundary(float x, float s, float q)
{
    const uint32_t mb = (__float_as_uint(fabsf(q)) + 4u) & ~0x7FFFFu;  // the nearest such m
    const float m = __uint_as_float(mb);
    const float e = fmaf(-s, m, fabsf(x));                                  // |x| - s*m, exact
    const float h = s * __uint_as_float((mb & 0x7F800000u) - (24u << 23));  // s * ulp(m) / 2
    const float t = e > h ? __uint_as_float(mb + 1u) : (e < -h ? __uint_as_float(mb - 1u) : m);
    return copysignf(t, x);
}

__device__ __forceinline__ uint32_t quant4(uint32_t a, uint32_t b, float s, float r)
{
    // bf16 pairs a = (x0, x1), b = (x2, x3) -> codes x0 | x1 << 8 | x2 << 16 | x3 << 24
    const float x[4] = {bf16lo_to_f32(a), bf16hi_to_f32(a), bf16lo_to_f32(b), bf16hi_to_f32(b)};
    float q[4];
    bool near = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[i] = x[i] * r;
        near = near || near_e4m3_boundary(q[i]);
    }
    // rare (about 1e-4 of the calls): resolve in a branch the warp takes together
    if (__any_sync(__activemask(), near)) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (near_e4m3_boundary(q[i])) q[i] = resolve_near_boundary(x[i], s, q[i]);
    }
    return static_cast<uint32_t>(f32x2_to_e4m3x2(q[0], q[1])) |
           (static_cast<uint32_t>(f32x2_to_e4m3x2(q[2], q[3])) << 16);
}

constexpr int kAppendMaxHeadsPerWarp = 8;


// Token t of the call, kv heads h0 .. h0 + nh - 1, by one warp
template <int D>
__device__ __forceinline__ void append_fp8_token(const AppendParams &p, const int32_t t,
                                                 const int32_t h0, const int32_t nh, const int lane,
                                                 const bool skip_whole = false)
{
    constexpr int kPerHead = D / 4;                          // 4-byte words per head and tensor
    constexpr int kPerLane = (kPerHead + 31) / 32;
    constexpr int kMaxHeads = kAppendMaxHeadsPerWarp;
    const int32_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) return;
    if (slot >= p.num_slots) {
        if (lane == 0) report(p.status, PKV_DEV_BAD_SLOT);
        return;
    }
    const int32_t off = slot & 15;
    const int32_t lead = t - off;  // the block's first token, if the block is whole
    bool mine = true;
    if (lane < 16) {
        const int32_t u = lead + lane;
        mine = u >= 0 && u < p.num_tokens && __ldg(p.slot_mapping + u) == slot - off + lane;
    }
    const bool whole = __all_sync(0xffffffffu, mine);
    if (whole && skip_whole) return;  // the block's tile is written whole elsewhere
    const int64_t tok_stride = static_cast<int64_t>(p.hkv) * D;  // elements per token row set
    const uint16_t *knew = static_cast<const uint16_t *>(p.k_new);
    const uint16_t *vnew = static_cast<const uint16_t *>(p.v_new);
    const uint32_t *krow = reinterpret_cast<const uint32_t *>(knew + t * tok_stride);
    const uint32_t *vrow = reinterpret_cast<const uint32_t *>(vnew + t * tok_stride);
    // whole blocks: this warp's token quad cq of V words, dims (off % 4) * D/4 ..
    // (formed only for whole blocks, whose 16 tokens all exist)
    const int cq = off >> 2;
    const int64_t q0 = whole ? (lead + 2 * cq) * tok_stride : 0;
    const uint16_t *vq0 = vnew + q0;
    const uint16_t *vq1 = vnew + (whole ? q0 + tok_stride : 0);
    const uint16_t *vq2 = vnew + (whole ? q0 + 8 * tok_stride : 0);
    const uint16_t *vq3 = vnew + (whole ? q0 + 9 * tok_stride : 0);
    uint8_t *kt0 = static_cast<uint8_t *>(p.k_pool) + static_cast<int64_t>(slot >> 4) * p.hkv * (16 * D);
    uint8_t *vt0 = static_cast<uint8_t *>(p.v_pool) + static_cast<int64_t>(slot >> 4) * p.hkv * (16 * D);
    // V byte of (token off, dim d): (d/32)*512 + ((d%8)*4 + cv)*16 + ((d%32)/8)*4 + jv
    const int32_t cv = (off & 7) >> 1, jv = (off & 1) + 2 * (off >> 3);
    const float kr_s = __frcp_rn(p.k_scale), vr_s = __frcp_rn(p.v_scale);
    // every head's loads first (up to kMaxHeads per warp), then the codes:
    // the loads of all heads are in flight together
    uint32_t kin[kMaxHeads][kPerLane][2], vin[kMaxHeads][kPerLane][2];
#pragma unroll
    for (int hh = 0; hh < kMaxHeads; ++hh) {
        const int h = h0 + hh;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            kin[hh][i][0] = kin[hh][i][1] = vin[hh][i][0] = vin[hh][i][1] = 0;
            const int w = lane + 32 * i;
            if (hh >= nh || (kPerHead < 32 && w >= kPerHead)) continue;
            const int u = w >> 2, kk = w & 3, grp = u >> 2, c = u & 3;
            const int d0 = grp * 64 + kk * 16 + 2 * c;  // dims d0, d0+1, d0+8, d0+9
            const uint32_t *kr = krow + h * (D / 2);
            kin[hh][i][0] = __ldg(kr + d0 / 2);
            kin[hh][i][1] = __ldg(kr + d0 / 2 + 4);
            if (whole) {
                // V words of the block's tokens {2cq, 2cq+1, 2cq+8, 2cq+9}:
                // lanes read consecutive dims of the same four rows
                const int e = h * D + (off & 3) * kPerHead + w;
                vin[hh][i][0] = static_cast<uint32_t>(__ldg(vq0 + e)) |
                                (static_cast<uint32_t>(__ldg(vq1 + e)) << 16);
                vin[hh][i][1] = static_cast<uint32_t>(__ldg(vq2 + e)) |
                                (static_cast<uint32_t>(__ldg(vq3 + e)) << 16);
            } else {
                const uint32_t *vr = vrow + h * (D / 2);
                vin[hh][i][0] = __ldg(vr + d0 / 2);
                vin[hh][i][1] = __ldg(vr + d0 / 2 + 4);
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < kMaxHeads; ++hh) {
        const int h = h0 + hh;
        uint8_t *ktile = kt0 + h * (16 * D);
        uint8_t *vtile = vt0 + h * (16 * D);
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int w = lane + 32 * i;
            if (hh >= nh || (kPerHead < 32 && w >= kPerHead)) continue;
            // K run (64-dim group grp, pair class c), 16-dim step kk
            const int u = w >> 2, kk = w & 3, grp = u >> 2, c = u & 3;
            const int d0 = grp * 64 + kk * 16 + 2 * c;
            *reinterpret_cast<uint32_t *>(ktile + grp * 1024 + (off >> 3) * 512 +
                                          ((off & 7) * 4 + c) * 16 + kk * 4) =
                quant4(kin[hh][i][0], kin[hh][i][1], p.k_scale, kr_s);
            const uint32_t vc = quant4(vin[hh][i][0], vin[hh][i][1], p.v_scale, vr_s);
            if (whole) {
                const int d = (off & 3) * kPerHead + w;
                const int g32 = d >> 5, jn = (d & 31) >> 3, n = d & 7;
                *reinterpret_cast<uint32_t *>(vtile + g32 * 512 + (4 * n + cq) * 16 + jn * 4) = vc;
            } else {
                const int32_t vd[4] = {d0, d0 + 1, d0 + 8, d0 + 9};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int32_t dd = vd[j];
                    vtile[(dd >> 5) * 512 + ((dd & 7) * 4 + cv) * 16 + ((dd & 31) >> 3) * 4 + jv] =
                        static_cast<uint8_t>(vc >> (8 * j));
                }
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256) append_fp8_kernel(AppendParams p)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int32_t groups = p.hkv / p.heads_per_warp;
    const int64_t items = static_cast<int64_t>(p.num_tokens) * groups;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < items;
         i += nwarps)
        append_fp8_token<D>(p, static_cast<int32_t>(i / groups),
                            static_cast<int32_t>(i % groups) * p.heads_per_warp, p.heads_per_warp, lane);
}

// Bulk FP8 append: one CTA per window of 16 tokens of the call.  A block
// whose 16 tokens come in order from the call (its lead token, the one at
// slot offset 0, lies in the window) is written as whole tiles: for each run
// of HG kv heads, the 16 tokens' bf16 K and V rows are staged in shared memory
// (16-byte asynchronous copies, rows padded to 2D + 16 bytes so that the
// reads below hit distinct banks), then every thread forms whole 16-byte
// chunks of the tiles in the tiles' byte order (a K chunk: one token, the 16
// dims of one pair class over four 16-dim steps; a V chunk: one dim of four
// tokens over four 8-dim steps) and stores them with coalesced 16-byte stores.
// Tokens of blocks that are not whole (ragged chunk ends) are then written
// by the per-token path, one warp per token.  At most one lead lies in a
// window (a whole block spans 16 tokens of the call).
constexpr int kAppendWindow = 16;

template <int D>
struct AppendWin {
    static constexpr int kHG = 512 / D;          // kv heads per staging round
    static constexpr int kRowB = 2 * D + 16;     // padded bytes of one (head, token) row
    static constexpr int kTensorB = kHG * kAppendWindow * kRowB;
    static constexpr int kSmem = 2 * kTensorB;   // K and V
};

template <int D>
__global__ void __launch_bounds__(256) append_fp8_window_kernel(AppendParams p)
{
    using W = AppendWin<D>;
    constexpr int HG = W::kHG;
    extern __shared__ __align__(16) uint8_t sm[];
    __shared__ int32_t s_lead;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t t0 = blockIdx.x * kAppendWindow;
    // the window's lead of a whole block, if any: thread k checks token
    // t0 + k/16 against the slot of token t0 + k/16 + k%16
    if (threadIdx.x == 0) s_lead = -1;
    __syncthreads();
    {
        const int32_t tw = t0 + (threadIdx.x >> 4), i = threadIdx.x & 15;
        bool ok = false;
        if (tw < p.num_tokens && tw + i < p.num_tokens) {
            const int32_t s0 = __ldg(p.slot_mapping + tw);
            ok = s0 >= 0 && s0 < p.num_slots && (s0 & 15) == 0 && __ldg(p.slot_mapping + tw + i) == s0 + i;
        }
        const uint32_t m = __ballot_sync(0xffffffffu, ok);
        const uint32_t mine = (m >> (lane & 16)) & 0xFFFFu;
        if (i == 0 && mine == 0xFFFFu) s_lead = tw;
    }
    __syncthreads();
    const int32_t lead = s_lead;
    if (lead >= 0) {
        const int32_t blk = __ldg(p.slot_mapping + lead) >> 4;
        const float ks = p.k_scale, vs = p.v_scale;
        const float kr = __frcp_rn(ks), vr = __frcp_rn(vs);
        for (int32_t h0 = 0; h0 < p.hkv; h0 += HG) {
            const int nh = min(HG, p.hkv - h0);
            // stage: tensor x (head, token) rows of D/8 16-byte chunks
            constexpr int kRowChunks = D / 8;
            constexpr int kChunks = 2 * HG * kAppendWindow * kRowChunks;
            for (int q = threadIdx.x; q < kChunks; q += blockDim.x) {
                const int tensor = q / (HG * kAppendWindow * kRowChunks);
                const int rr = q % (HG * kAppendWindow * kRowChunks);
                const int row = rr / kRowChunks, col = rr % kRowChunks;
                const int hh = row / kAppendWindow, tok = row % kAppendWindow;
                if (hh >= nh) continue;
                const uint8_t *src = static_cast<const uint8_t *>(tensor ? p.v_new : p.k_new) +
                                     ((static_cast<int64_t>(lead + tok) * p.hkv + h0 + hh) * D) * 2 +
                                     col * 16;
                const uint32_t dst = smem_u32(sm + tensor * W::kTensorB + row * W::kRowB + col * 16);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
            }
            asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
            __syncthreads();
            // chunks: per head D of K then D of V, 16 bytes each
            for (int q = threadIdx.x; q < nh * 2 * D; q += blockDim.x) {
                const int hh = q / (2 * D), r = q % (2 * D);
                const bool is_v = r >= D;
                const int c = is_v ? r - D : r;
                const uint8_t *base = sm + (is_v ? W::kTensorB : 0) + hh * kAppendWindow * W::kRowB;
                uint32_t w4[4];
                if (!is_v) {
                    // byte 16c of the K tile: c = grp*64 + half*32 + t8*4 + cc; token
                    // half*8 + t8, words kk: dims grp*64 + 16kk + 2cc + {0, 1, 8, 9}
                    const int grp = c >> 6, tok = ((c >> 5) & 1) * 8 + ((c >> 2) & 7), cc = c & 3;
                    const uint8_t *rowp = base + tok * W::kRowB;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int d0 = grp * 64 + kk * 16 + 2 * cc;
                        const uint32_t a = *reinterpret_cast<const uint32_t *>(rowp + d0 * 2);
                        const uint32_t b = *reinterpret_cast<const uint32_t *>(rowp + (d0 + 8) * 2);
                        w4[kk] = quant4(a, b, ks, kr);
                    }
                } else {
                    // byte 16c of the V tile: c = g32*32 + n*4 + cq; words jn: dim
                    // g32*32 + 8jn + n of tokens 2cq, 2cq + 1, 2cq + 8, 2cq + 9
                    const int g32 = c >> 5, n = (c >> 2) & 7, cq = c & 3;
                    const uint16_t *r0 = reinterpret_cast<const uint16_t *>(base + (2 * cq) * W::kRowB);
                    const uint16_t *r1 = reinterpret_cast<const uint16_t *>(base + (2 * cq + 1) * W::kRowB);
                    const uint16_t *r8 = reinterpret_cast<const uint16_t *>(base + (2 * cq + 8) * W::kRowB);
                    const uint16_t *r9 = reinterpret_cast<const uint16_t *>(base + (2 * cq + 9) * W::kRowB);
#pragma unroll
                    for (int jn = 0; jn < 4; ++jn) {
                        const int d = g32 * 32 + jn * 8 + n;
                        const uint32_t a = static_cast<uint32_t>(r0[d]) | (static_cast<uint32_t>(r1[d]) << 16);
                        const uint32_t b = static_cast<uint32_t>(r8[d]) | (static_cast<uint32_t>(r9[d]) << 16);
                        w4[jn] = quant4(a, b, vs, vr);
                    }
                }
                uint8_t *tile = static_cast<uint8_t *>(is_v ? p.v_pool : p.k_pool) +
                                (static_cast<int64_t>(blk) * p.hkv + h0 + hh) * (16 * D);
                __stcs(reinterpret_cast<uint4 *>(tile) + c, make_uint4(w4[0], w4[1], w4[2], w4[3]));
            }
            __syncthreads();  // the staging rows are refilled by the next round
        }
    }
    // tokens of the window whose block is not whole: one warp per token
    for (int32_t i = warp; i < kAppendWindow; i += blockDim.x >> 5) {
        const int32_t t = t0 + i;
        if (t >= p.num_tokens) break;
        for (int32_t h0 = 0; h0 < p.hkv; h0 += kAppendMaxHeadsPerWarp)
            append_fp8_token<D>(p, t, h0, min(kAppendMaxHeadsPerWarp, p.hkv - h0), lane, true);
    }
}

cudaError_t launch_append_fp8(const AppendParams &p, cudaStream_t stream)
{
    if (p.num_tokens == 0 || p.hkv == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (p.head_dim != 64 && p.head_dim != 128 && p.head_dim != 256) return cudaErrorInvalidValue;
    // bulk appends (a prefill chunk, a whole context): whole-tile windows
    if (static_cast<int64_t>(p.num_tokens) >= 8ll * sms) {
        const unsigned grid = static_cast<unsigned>((p.num_tokens + kAppendWindow - 1) / kAppendWindow);
        cudaError_t err;
        prof_begin(PKV_KERNEL_APPEND, stream);
        switch (p.head_dim) {
        case 64:
            err = launch_pdl(append_fp8_window_kernel<64>, dim3(grid), dim3(256), AppendWin<64>::kSmem, stream, p);
            break;
        case 128:
            err = launch_pdl(append_fp8_window_kernel<128>, dim3(grid), dim3(256), AppendWin<128>::kSmem, stream, p);
            break;
        default:
            err = launch_pdl(append_fp8_window_kernel<256>, dim3(grid), dim3(256), AppendWin<256>::kSmem, stream, p);
            break;
        }
        prof_end(PKV_KERNEL_APPEND, stream);
        return err;
    }
    // a warp takes all kv heads of a token (the slot checks once per token)
    // unless that leaves fewer than 32 warps per SM (a decode step's few
    // tokens): then fewer heads per warp, down to one
    AppendParams q = p;
    q.heads_per_warp = p.hkv;
    while (q.heads_per_warp % 2 == 0 &&
           (q.heads_per_warp > kAppendMaxHeadsPerWarp ||
            static_cast<int64_t>(p.num_tokens) * (p.hkv / q.heads_per_warp) < 32ll * sms))
        q.heads_per_warp /= 2;
    // an odd head count above the cap: one head per warp
    if (q.heads_per_warp > kAppendMaxHeadsPerWarp) q.heads_per_warp = 1;
    const int64_t warps = static_cast<int64_t>(p.num_tokens) * (p.hkv / q.heads_per_warp);
    // a grid-stride loop: at most 8 CTAs of 8 warps per SM
    const int64_t blocks = std::min<int64_t>((warps + 7) / 8, static_cast<int64_t>(sms) * 8);
    auto kern = p.head_dim == 64 ? append_fp8_kernel<64>
                                 : (p.head_dim == 128 ? append_fp8_kernel<128> : append_fp8_kernel<256>);
    prof_begin(PKV_KERNEL_APPEND, stream);
    const cudaError_t err = launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, q);
    prof_end(PKV_KERNEL_APPEND, stream);
    return err;
}

}  // namespace pkv
