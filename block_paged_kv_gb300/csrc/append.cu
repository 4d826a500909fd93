// Append of new K/V rows into their pool slots ("perf.md", paged knob table:
// the graph-native paged K/V write, MLX_PAGED_NATIVE_KV_WRITE).
//
// One thread moves one 16-byte vector of one (token, kv head) row for both K
// and V: two 16-byte loads and two 16-byte stores, all coalesced within the
// row (a bf16 head_dim-128 row is 16 vectors).  HBM bound: the algorithmic
// traffic is 2 x (read + write) x num_tokens x Hkv x head_dim x elem bytes plus
// 4 bytes of slot per token.
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
// float32 quotient x / scale (IEEE division, round to nearest even,
// saturating).  One thread per (token, kv head, 64-dim group, pair class c)
// quantizes the 16 dims kk*16 + {2c, 2c+1, 2c+8, 2c+9} (kk = 0..3) of the K
// row and of the V row: in the K tile they are one 16-byte run (one store);
// in the V tile each is a byte of its own (V is stored token-minor).
__global__ void __launch_bounds__(256) append_fp8_kernel(AppendParams p)
{
    pdl_wait();
    pdl_trigger();
    const int32_t units = p.head_dim / 16;  // (group, c) per row
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.hkv * units;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int32_t u = static_cast<int32_t>(idx % units);
    const int64_t th = idx / units;
    const int32_t h = static_cast<int32_t>(th % p.hkv);
    const int32_t t = static_cast<int32_t>(th / p.hkv);
    const int32_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) return;
    if (slot >= p.num_slots) {
        if (h == 0 && u == 0) report(p.status, PKV_DEV_BAD_SLOT);
        return;
    }
    const int32_t grp = u >> 2, c = u & 3;
    const int32_t blk = slot >> 4, off = slot & 15;
    const int64_t tile = (static_cast<int64_t>(blk) * p.hkv + h) * (16 * p.head_dim);
    const int64_t row = th * p.head_dim;
    const uint32_t *krow = reinterpret_cast<const uint32_t *>(
        static_cast<const uint16_t *>(p.k_new) + row);
    const uint32_t *vrow = reinterpret_cast<const uint32_t *>(
        static_cast<const uint16_t *>(p.v_new) + row);
    uint8_t *vtile = static_cast<uint8_t *>(p.v_pool) + tile;
    // V byte of (token off, dim d): (d/32)*512 + ((d%8)*4 + cv)*16 + ((d%32)/8)*4 + jv
    const int32_t cv = (off & 7) >> 1, jv = (off & 1) + 2 * (off >> 3);
    uint32_t kw[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int32_t d0 = grp * 64 + kk * 16 + 2 * c;  // dims d0, d0+1, d0+8, d0+9
        const uint32_t ka = __ldg(krow + d0 / 2), kb = __ldg(krow + d0 / 2 + 4);
        const uint32_t va = __ldg(vrow + d0 / 2), vb = __ldg(vrow + d0 / 2 + 4);
        const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_to_f32(ka), p.k_scale),
                                            __fdiv_rn(bf16hi_to_f32(ka), p.k_scale));
        const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_to_f32(kb), p.k_scale),
                                            __fdiv_rn(bf16hi_to_f32(kb), p.k_scale));
        kw[kk] = lo | (hi << 16);
        const float vx[4] = {bf16lo_to_f32(va), bf16hi_to_f32(va), bf16lo_to_f32(vb),
                             bf16hi_to_f32(vb)};
        const int32_t vd[4] = {d0, d0 + 1, d0 + 8, d0 + 9};
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const uint16_t codes = f32x2_to_e4m3x2(__fdiv_rn(vx[e], p.v_scale),
                                                   __fdiv_rn(vx[e + 1], p.v_scale));
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int32_t d = vd[e + i];
                vtile[(d >> 5) * 512 + ((d & 7) * 4 + cv) * 16 + ((d & 31) >> 3) * 4 + jv] =
                    static_cast<uint8_t>(codes >> (8 * i));
            }
        }
    }
    // K byte of (token off, dim d): (d/64)*1024 + (off/8)*512 + ((off%8)*4 + c)*16 + kk*4 + j
    *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.k_pool) + tile + grp * 1024 +
                               (off >> 3) * 512 + ((off & 7) * 4 + c) * 16) =
        make_uint4(kw[0], kw[1], kw[2], kw[3]);
}

cudaError_t launch_append_fp8(const AppendParams &p, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(p.num_tokens) * p.hkv * (p.head_dim / 16);
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    prof_begin(PKV_KERNEL_APPEND, stream);
    const cudaError_t err = launch_pdl(append_fp8_kernel, dim3(static_cast<unsigned>(blocks)),
                                       dim3(256), 0, stream, p);
    prof_end(PKV_KERNEL_APPEND, stream);
    return err;
}

}  // namespace pkv
