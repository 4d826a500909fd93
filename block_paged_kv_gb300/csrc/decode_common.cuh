// Per-row key ranges and split bookkeeping shared by the decode kernels and
// the combine kernel, so that both sides agree on which partial slots exist.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct RowRange {
    int32_t L;        // clamped sequence length
    int32_t C;        // queries of the row (1 for decode), at positions L - C .. L - 1
    int32_t q0;       // index of the row's first query in the packed q / out
    int32_t lo;       // first position any of its queries attends
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
    rr.C = 1;
    rr.q0 = r;
    if (p.cu_q_lens != nullptr) {
        const int32_t c0 = __ldg(p.cu_q_lens + r), c1 = __ldg(p.cu_q_lens + r + 1);
        int32_t C = c1 - c0;
        if (c0 < 0 || C < 0 || C > p.max_q || C > L) {
            if (report_bad) report(p.status, PKV_DEV_BAD_LEN);
            C = c0 < 0 || C < 0 ? 0 : min(min(C, p.max_q), L);
        }
        rr.C = C;
        rr.q0 = c0 < 0 ? 0 : c0;
    }
    // the first query (position L - C) reaches back furthest
    rr.lo = p.window > 0 ? max(0, L - rr.C + 1 - p.window) : 0;
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

// Partial slots of query t of row r (t = 0 for decode), q head h.
__device__ __forceinline__ size_t partial_index(const DecodeParams &p, int32_t r, int32_t h,
                                                int32_t slot, int32_t t = 0)
{
    return ((static_cast<size_t>(r) * p.max_q + t) * p.hq + h) * p.plan.nslot + slot;
}

}  // namespace pkv
