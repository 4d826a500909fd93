// Per-row key ranges and split bookkeeping shared by the decode kernels and
// the combine kernel, so that both sides agree on which partial slots exist.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct RowRange {
    int32_t L;        // clamped sequence length
    int32_t lo;       // first attended position
    int32_t b_first;  // first block of the row's own (suffix) splits
    int32_t b_end;    // one past the last block holding a position < L
    int32_t grp;      // shared-prefix group, -1 = none
    int32_t P;        // prefix blocks of the group (0 = none)
};

__device__ __forceinline__ int32_t ceil_div_i(int32_t a, int32_t b) { return (a + b - 1) / b; }

// Key range of row r.  Lengths outside [0, max_len] are clamped (and reported
// when `report_bad`); an out-of-range group id drops the row from prefix
// sharing; a prefix longer than the plan's bound is cut to it.
__device__ __forceinline__ RowRange row_range(const DecodeParams &p, int32_t r, bool report_bad)
{
    RowRange rr;
    int32_t L = __ldg(p.seq_lens + r);
    if (L < 0 || L > p.max_len) {
        if (report_bad) report(p.status, PKV_DEV_BAD_LEN);
        L = L < 0 ? 0 : p.max_len;
    }
    rr.L = L;
    rr.lo = p.window > 0 ? max(0, L - p.window) : 0;
    rr.b_first = rr.lo / p.block_size;
    rr.b_end = ceil_div_i(L, p.block_size);
    rr.grp = -1;
    rr.P = 0;
    if (p.group_of_row != nullptr) {
        int32_t grp = __ldg(p.group_of_row + r);
        if (grp >= p.num_groups) {
            if (report_bad) report(p.status, PKV_DEV_BAD_PREFIX);
            grp = -1;
        }
        if (grp >= 0) {
            int32_t P = __ldg(p.prefix_blocks + grp);
            const int32_t pmax = p.plan.prefix_max;
            if (P < 0 || P > pmax) {
                if (report_bad) report(p.status, PKV_DEV_BAD_PREFIX);
                P = P < 0 ? 0 : pmax;
            }
            rr.grp = grp;
            rr.P = P;
            rr.b_first = max(rr.b_first, P);
        }
    }
    return rr;
}

__device__ __forceinline__ int32_t row_suffix_splits(const DecodeParams &p, const RowRange &rr)
{
    return rr.b_end > rr.b_first ? ceil_div_i(rr.b_end - rr.b_first, p.plan.split_blocks) : 0;
}

__device__ __forceinline__ int32_t row_prefix_splits(const DecodeParams &p, const RowRange &rr)
{
    return rr.grp >= 0 ? ceil_div_i(rr.P, p.plan.prefix_split_blocks) : 0;
}

__device__ __forceinline__ size_t partial_index(const DecodeParams &p, int32_t r, int32_t h,
                                                int32_t slot)
{
    return (static_cast<size_t>(r) * p.hq + h) * p.plan.nslot + slot;
}

}  // namespace pkv
