"""The seeded input generator: published SplitMix64 values, bf16 rounding,
distribution sanity and the structure of the five workloads (CPU)."""
import numpy as np

import pkv_inputs as gen


def test_splitmix64_reference_value():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF
    assert int(gen.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF
    # counter-based: word i is independent of how the stream is chunked
    a = gen.splitmix64(12345, 0, 10)
    b = np.concatenate([gen.splitmix64(12345, 0, 4), gen.splitmix64(12345, 4, 6)])
    assert np.array_equal(a, b)


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7 + 2 ** -8, -2.5, 0.0],
                 dtype=np.float32)
    assert gen.bf16_bits(x).tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F82, 0xC020, 0x0000]
    v = gen.normal_f32(1, "x", 1000)
    assert np.array_equal(gen.bf16_to_f32(gen.bf16_bits(gen.bf16_to_f32(gen.bf16_bits(v)))),
                          gen.bf16_to_f32(gen.bf16_bits(v)))


def test_normal_moments_and_permutation():
    v = gen.normal_f32(3, "x", 200001).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.var() - 1) < 0.01
    p = gen.permutation(5, "p", 1000)
    assert sorted(p.tolist()) == list(range(1000)) and not np.array_equal(p, np.arange(1000))


def test_tiny_workload_structure():
    w = gen.tiny_f32()
    assert w.seq_lens.tolist() == [37, 50] and w.num_blocks == 16
    assert w.block_tables.shape == (2, 4)
    assert np.array_equal(w.block_tables[0, :2], w.block_tables[1, :2])  # 2-block shared prefix
    ids = w.block_tables[w.block_tables >= 0]
    assert len(set(ids.tolist())) == 5
    assert w.new_pos.tolist() == [36, 49]
    assert w.dtype == "f32" and w.q.shape == (2, 4, 64)


def test_shared_prefix_workload_structure():
    w = gen.shared_prefix_b32(batch=8, max_suffix=300)
    assert np.all(w.block_tables[:, :64] == w.block_tables[0, :64])
    used = w.block_tables[w.block_tables >= 0]
    assert len(set(used.tolist())) == w.num_blocks  # pool sized to the total
    assert np.all((w.seq_lens - 1025 >= 0) & (w.seq_lens - 1025 <= 300))


def test_sliding_workload_structure():
    full, sl = gen.long_two_groups(batch=2, context=1024, window=64)
    lo = 1024 - 64
    assert np.all(sl.block_tables[:, :lo // 16] == -1)
    assert np.all(sl.block_tables[:, lo // 16:] >= 0)
    assert sl.num_blocks == 2 * 5 and full.num_blocks == 2 * 64


def test_prefill_workload_structure():
    w = gen.chunked_prefill(batch=2, chunk=32, prefix=64)
    assert w.cu_q_lens.tolist() == [0, 32, 64] and w.q.shape == (64, 32, 128)
    assert w.seq_lens.tolist() == [96, 96] and w.new_pos[:3].tolist() == [64, 65, 66]
