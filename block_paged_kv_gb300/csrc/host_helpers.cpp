// Host helpers of the C ABI: slot mapping, its debug check and shared-prefix
// group derivation from block tables.  Plain C++ on host arrays.
#include <algorithm>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv.h"

extern "C" pkv_status pkv_slot_mapping_host(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                            int32_t batch, int32_t num_blocks, const int32_t *rows,
                                            const int32_t *positions, int32_t n, int32_t block_size,
                                            int32_t *slots_out)
{
    if (n < 0 || block_size <= 0 || batch < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (n > 0 && (rows == nullptr || positions == nullptr || slots_out == nullptr ||
                  block_tables == nullptr))
        return PKV_ERR_INVALID_ARG;
    bool all_ok = true;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t row = rows[i], pos = positions[i];
        int32_t slot = -1;
        if (row >= 0 && row < batch && pos >= 0) {
            const int32_t logical = pos / block_size;
            if (logical < max_blocks_per_seq) {
                const int32_t phys = block_tables[static_cast<int64_t>(row) * max_blocks_per_seq + logical];
                if (phys >= 0 && phys < num_blocks &&
                    static_cast<int64_t>(phys) * block_size + block_size <= INT32_MAX)
                    slot = phys * block_size + (pos - logical * block_size);
            }
        }
        slots_out[i] = slot;
        all_ok = all_ok && slot >= 0;
    }
    return all_ok ? PKV_OK : PKV_ERR_INVALID_ARG;
}

extern "C" pkv_status pkv_slot_mapping_check_host(const int32_t *slots, int32_t n,
                                                  int32_t num_blocks, int32_t block_size,
                                                  int32_t *first_bad)
{
    if (first_bad != nullptr) *first_bad = -1;
    if (n < 0 || num_blocks <= 0 || block_size <= 0 || (n > 0 && slots == nullptr))
        return PKV_ERR_INVALID_ARG;
    const int64_t cap = static_cast<int64_t>(num_blocks) * block_size;
    std::unordered_set<int32_t> seen;
    seen.reserve(static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i) {
        const int32_t s = slots[i];
        if (s < 0) continue;  // skipped by the append
        if (static_cast<int64_t>(s) >= cap || !seen.insert(s).second) {
            if (first_bad != nullptr) *first_bad = i;
            return PKV_ERR_INVALID_ARG;
        }
    }
    return PKV_OK;
}

extern "C" int32_t pkv_prefix_groups_host(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *seq_lens, int32_t batch, int32_t block_size,
                                          int32_t *group_of_row, int32_t *prefix_blocks)
{
    if (batch < 0 || max_blocks_per_seq <= 0 || block_size <= 0) return -1;
    if (batch > 0 && (block_tables == nullptr || seq_lens == nullptr || group_of_row == nullptr ||
                      prefix_blocks == nullptr))
        return -1;
    auto table = [&](int32_t r) { return block_tables + static_cast<int64_t>(r) * max_blocks_per_seq; };
    // rows bucketed by their first physical block, buckets kept in order of
    // their lowest row
    std::unordered_map<int32_t, size_t> bucket_of_block;
    std::vector<std::vector<int32_t>> buckets;
    for (int32_t r = 0; r < batch; ++r) {
        group_of_row[r] = -1;
        const int32_t first = table(r)[0];
        if (first < 0) continue;
        auto it = bucket_of_block.find(first);
        if (it == bucket_of_block.end()) {
            bucket_of_block.emplace(first, buckets.size());
            buckets.push_back({r});
        } else {
            buckets[it->second].push_back(r);
        }
    }
    int32_t ngroups = 0;
    for (const auto &rows : buckets) {
        if (rows.size() < 2) continue;
        // common run against the bucket's first row, cut to full blocks
        const int32_t *lead = table(rows[0]);
        int32_t run = max_blocks_per_seq;
        for (const int32_t r : rows) {
            const int32_t *t = table(r);
            int32_t k = 0;
            const int32_t lim = std::min(run, std::max(0, seq_lens[r]) / block_size);
            while (k < lim && t[k] == lead[k]) ++k;
            run = k;
        }
        if (run <= 0) continue;
        for (const int32_t r : rows) group_of_row[r] = ngroups;
        prefix_blocks[ngroups++] = run;
    }
    return ngroups;
}
