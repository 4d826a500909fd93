"""The byte counts behind bench.py's throughput and roofline figures (CPU).

The decode step's algorithmic bytes are the K/V rows of every attended token
slot, each counted once: a prefix block that all rows share through their
block tables is read once by the read-once path, so it is counted once too.
Here that count is taken slot by slot from the workload's own block tables and
compared with the formula the bench uses."""
import os
import sys

import numpy as np

import pkv_inputs as gen

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _attended_slots(w):
    slots = set()
    for r in range(w.batch):
        for pos in range(int(w.seq_lens[r])):
            slots.add((int(w.block_tables[r, pos // w.block_size]), pos % w.block_size))
    return slots


def test_step_bytes_count_each_attended_slot_once():
    w = gen.shared_prefix_b32(batch=8, max_suffix=300)
    per_token = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes  # K and V of every kv head
    slots = _attended_slots(w)
    total, split = bench.workload_bytes(w)
    assert total == len(slots) * per_token
    # the split CTAs' share: everything past the shared prefix
    assert split == (len(slots) - w.shared_prefix_tokens) * per_token
    # without sharing every row would read the prefix itself
    private = int(np.sum(w.seq_lens.astype(np.int64))) * per_token
    assert private - total == (w.batch - 1) * w.shared_prefix_tokens * per_token


def test_headline_step_bytes():
    # 32 rows: the 1024-token prefix once, then each row's suffix and the
    # token it appends; 4096 bytes per token (K and V, 8 kv heads x 128 x bf16)
    suffixes = gen.shared_prefix_suffix_lens(1002, 32, 7168)
    tokens = 1024 + sum(s + 1 for s in suffixes)
    assert tokens - 1024 == 124682  # the tokens a bulk append of the suffixes writes
    assert tokens * 4096 == 514891776


def test_job_rate_sums_ranks():
    # units per rank and step x ranks x steps / slowest rank's time
    assert bench.job_rate(1000, 2, 4.0, 8) == 1000 * 2 * 8 / 4e-3
