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
// division, r = the correctly rounded reciprocal of s.
//
// q0 = RN(x * r) lies within one ulp of x / s (the rounding of the product
// and r's own half ulp).  One correction step then gives the correctly
// rounded quotient: e = x - s * q0 is exact (one fused multiply-add), and
// RN(q0 + e * r) = RN(x / s) when r = RN(1/s) and q0 is within one ulp, in
// the normal range (Markstein's theorem on the final step of an FMA
// division: P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  The step is
// taken where the last ulp can change the E4M3 code, 2^-11 <= |q0| <= 512:
// below, the code is a zero of x's sign; above, E4M3 saturates (448); NaN
// stays NaN.  Checked against the IEEE quotient on every bf16 input for
// thousands of scales, codes compared, and against the oracle's codes in the
// GPU tests.
__device__ __forceinline__ float e4m3_quotient(float x, float s, float r)
{
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(-s, q0, x);
    const float q1 = __fmaf_rn(e, r, q0);
    const uint32_t a = __float_as_uint(q0) & 0x7FFFFFFFu;
    return (a - 0x3A000000u) <= 0x0A000000u ? q1 : q0;  // 2^-11 .. 512 as bits
}

__device__ __forceinline__ uint32_t quant4(uint32_t a, uint32_t b, float s, float r)
{
    // bf16 pairs a = (x0, x1), b = (x2, x3) -> codes x0 | x1 << 8 | x2 << 16 | x3 << 24
    const float q0 = e4m3_quotient(bf16lo_to_f32(a), s, r);
    const float q1 = e4m3_quotient(bf16hi_to_f32(a), s, r);
    const float q2 = e4m3_quotient(bf16lo_to_f32(b), s, r);
    const float q3 = e4m3_quotient(bf16hi_to_f32(b), s, r);
    return static_cast<uint32_t>(f32x2_to_e4m3x2(q0, q1)) |
           (static_cast<uint32_t>(f32x2_to_e4m3x2(q2, q3)) << 16);
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
    static constexpr int kSmem = 2 * kTensorB;   // K and V of one staging round
    static constexpr int kLaunchSmem = 2 * kSmem;  // two rounds in flight
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
        const int ngroups = (p.hkv + HG - 1) / HG;
        // staging round g (kv heads g*HG ..) into buffer g % 2: 16-byte
        // asynchronous copies of the (head, token) rows of K and V
        auto stage = [&](int g) {
            const int h0 = g * HG, nh = min(HG, p.hkv - h0);
            uint8_t *buf = sm + (g & 1) * W::kSmem;
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
                const uint32_t dst = smem_u32(buf + tensor * W::kTensorB + row * W::kRowB + col * 16);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        stage(0);
        if (ngroups > 1) stage(1);
        for (int g = 0; g < ngroups; ++g) {
            if (g + 1 < ngroups)
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            else
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            __syncthreads();
            const int h0 = g * HG, nh = min(HG, p.hkv - h0);
            const uint8_t *buf = sm + (g & 1) * W::kSmem;
            // per head: D items of one K chunk, then D/2 items of two V chunks
            // (dims n and n + 1 share their 4-byte shared-memory reads)
            constexpr int kItems = D + D / 2;
            for (int q = threadIdx.x; q < nh * kItems; q += blockDim.x) {
                const int hh = q / kItems, r = q % kItems;
                if (r < D) {
                    // byte 16c of the K tile: c = grp*64 + half*32 + t8*4 + cc; token
                    // half*8 + t8, words kk: dims grp*64 + 16kk + 2cc + {0, 1, 8, 9}
                    const int c = r;
                    const int grp = c >> 6, tok = ((c >> 5) & 1) * 8 + ((c >> 2) & 7), cc = c & 3;
                    const uint8_t *rowp = buf + (hh * kAppendWindow + tok) * W::kRowB;
                    uint32_t w4[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int d0 = grp * 64 + kk * 16 + 2 * cc;
                        const uint32_t a = *reinterpret_cast<const uint32_t *>(rowp + d0 * 2);
                        const uint32_t b = *reinterpret_cast<const uint32_t *>(rowp + (d0 + 8) * 2);
                        w4[kk] = quant4(a, b, ks, kr);
                    }
                    uint8_t *tile = static_cast<uint8_t *>(p.k_pool) +
                                    (static_cast<int64_t>(blk) * p.hkv + h0 + hh) * (16 * D);
                    __stcs(reinterpret_cast<uint4 *>(tile) + c, make_uint4(w4[0], w4[1], w4[2], w4[3]));
                } else {
                    // bytes 16c and 16(c + 4) of the V tile, c = g32*32 + n*4 + cq, n
                    // even: words jn of chunk c hold dim g32*32 + 8jn + n of tokens
                    // 2cq, 2cq + 1, 2cq + 8, 2cq + 9, those of chunk c + 4 dim + 1
                    const int v = r - D;
                    const int g32 = v >> 4, n = ((v >> 2) & 3) * 2, cq = v & 3;
                    const int c = g32 * 32 + n * 4 + cq;
                    const uint8_t *vb = buf + W::kTensorB + (hh * kAppendWindow + 2 * cq) * W::kRowB;
                    uint32_t w0[4], w1[4];
#pragma unroll
                    for (int jn = 0; jn < 4; ++jn) {
                        const int off = (g32 * 32 + jn * 8 + n) * 2;
                        const uint32_t t0 = *reinterpret_cast<const uint32_t *>(vb + off);
                        const uint32_t t1 = *reinterpret_cast<const uint32_t *>(vb + W::kRowB + off);
                        const uint32_t t8 = *reinterpret_cast<const uint32_t *>(vb + 8 * W::kRowB + off);
                        const uint32_t t9 = *reinterpret_cast<const uint32_t *>(vb + 9 * W::kRowB + off);
                        w0[jn] = quant4(__byte_perm(t0, t1, 0x5410), __byte_perm(t8, t9, 0x5410), vs, vr);
                        w1[jn] = quant4(__byte_perm(t0, t1, 0x7632), __byte_perm(t8, t9, 0x7632), vs, vr);
                    }
                    uint4 *tile = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.v_pool) +
                                                            (static_cast<int64_t>(blk) * p.hkv + h0 + hh) * (16 * D));
                    __stcs(tile + c, make_uint4(w0[0], w0[1], w0[2], w0[3]));
                    __stcs(tile + c + 4, make_uint4(w1[0], w1[1], w1[2], w1[3]));
                }
            }
            __syncthreads();  // buffer g % 2 is refilled by round g + 2
            if (g + 2 < ngroups) stage(g + 2);
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

template <int D>
static cudaError_t launch_append_window(const AppendParams &p, cudaStream_t stream)
{
    auto kern = append_fp8_window_kernel<D>;
    const int smem = AppendWin<D>::kLaunchSmem;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>((p.num_tokens + kAppendWindow - 1) / kAppendWindow);
    prof_begin(PKV_KERNEL_APPEND, stream);
    err = launch_pdl(kern, dim3(grid), dim3(256), smem, stream, p);
    prof_end(PKV_KERNEL_APPEND, stream);
    return err;
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
        switch (p.head_dim) {
        case 64: return launch_append_window<64>(p, stream);
        case 128: return launch_append_window<128>(p, stream);
        default: return launch_append_window<256>(p, stream);
        }
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
