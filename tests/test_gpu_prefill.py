"""GPU parity of the chunked prefill against the oracle (through the C ABI).

The chunk's K/V is appended first (paged_kv_append), then every query of the
chunk attends the paged prefix and the chunk causally.  Tolerances as for
decode: bf16 |gpu - ref| <= 2e-3 + 1e-2 |ref|; f32 1e-5 + 1e-5 |ref|.
"""
import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import (Dev, append, assert_appended_blocks_equal, assert_close, oracle_pools,
                      storage_bytes, to_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


def run_prefill(pkv, orc, w, samples=None, check_pool=True):
    d = Dev(w)
    slots = append(pkv, d)
    or_slots, kp, vp = oracle_pools(orc, w)
    assert np.array_equal(slots, or_slots)
    if check_pool:
        assert storage_bytes(d.k_pool) == kp.tobytes() and storage_bytes(d.v_pool) == vp.tobytes()
    else:
        assert_appended_blocks_equal(d, slots, kp, vp)
    max_q = int(np.max(np.diff(w.cu_q_lens)))
    out = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens,
                                            max_q, w.window, w.scale,
                                            max_seq_len=int(w.seq_lens.max()), status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0, int(d.status.item())
    got = to_f64(out)
    if samples is None:
        ref = orc.prefill(w.q, w.cu_q_lens, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window,
                          w.scale)
        return got, ref, d
    ref = _oracle_samples(orc, w, kp, vp, samples)
    rows = w.cu_q_lens[samples[:, 0]] + samples[:, 1]
    return got[rows, samples[:, 2]], ref, d


def _oracle_samples(orc, w, kp, vp, samples, chunk=64):
    """The oracle at (row, query, head) samples, chunks of them on a pool of
    host threads (the oracle's C calls release the interpreter lock)."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    def one(i):
        return orc.prefill(w.q, w.cu_q_lens, kp, vp, w.dtype, w.block_tables, w.seq_lens,
                           w.window, w.scale, samples=samples[i:i + chunk])

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        parts = list(ex.map(one, range(0, samples.shape[0], chunk)))
    return np.concatenate(parts)


def test_chunked_prefill_full_size(pkv, orc):
    # the oracle costs 5.6e11 FLOP over the whole call, so the outputs are
    # sampled: every query index of row 0 for one q head of each kv head
    # (a different head offset per kv head), the chunk's ends of every row,
    # and seeded (row, query, head) triples
    w = gen.chunked_prefill()
    u = gen.uniform_ints(5, "samples", 3 * 160, 0, 1 << 30)
    C = int(w.cu_q_lens[1] - w.cu_q_lens[0])
    G = w.num_q_heads // w.num_kv_heads
    samples = [[0, i, g * G + g % G] for g in range(w.num_kv_heads) for i in range(C)]
    samples += [[r, i, h] for r in range(w.batch) for i in (0, 1, 31, 32, C - 1)
                for h in (0, w.num_q_heads - 1)]
    samples += [[int(u[3 * k]) % w.batch, int(u[3 * k + 1]) % C, int(u[3 * k + 2]) % w.num_q_heads]
                for k in range(160)]
    samples = np.array(samples, dtype=np.int32)
    got, ref, _ = run_prefill(pkv, orc, w, samples=samples, check_pool=False)
    assert_close(got, ref, "bf16", "chunked prefill 4 x 512 vs 16384 prefix")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (16, 1)])
@pytest.mark.parametrize("window", [0, 50])
def test_ragged_shapes(pkv, orc, dtype, hq, hkv, window):
    w = gen.prefill_workload(seed=40 + hq + hkv + window, dtype=dtype, num_q_heads=hq,
                             num_kv_heads=hkv, head_dim=128,
                             prefix_lens=[0, 5, 130, 300], chunk_lens=[1, 47, 200, 129],
                             window=window)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, dtype, f"{dtype} prefill {hq}/{hkv} w{window}")


@pytest.mark.parametrize("d", [64, 256])
def test_f32_other_head_dims(pkv, orc, d):
    w = gen.prefill_workload(seed=60 + d, dtype="f32", num_q_heads=8, num_kv_heads=2, head_dim=d,
                             prefix_lens=[17, 64], chunk_lens=[9, 20], window=0)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "f32", f"f32 prefill d{d}")


def test_prefill_with_one_query_equals_decode(pkv):
    w = gen.prefill_workload(seed=70, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                             prefix_lens=[300, 1000, 31], chunk_lens=[1, 1, 1])
    d = Dev(w)
    append(pkv, d)
    pre = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 1,
                                            0, w.scale)
    dec = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale)
    torch.cuda.synchronize()
    assert_close(to_f64(pre), to_f64(dec), "bf16", "prefill C=1 vs decode")


def test_two_chunks_equal_one_chunk(pkv, orc):
    # the chunk of 200 queries prefilled at once, or as 120 then 80
    w = gen.prefill_workload(seed=71, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                             prefix_lens=[500], chunk_lens=[200])
    d = Dev(w)
    append(pkv, d)
    one = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 200,
                                            0, w.scale)
    first = pkv.paged_prefill_chunk_attention(
        d.q[:120].contiguous(), torch.tensor([0, 120], dtype=torch.int32, device="cuda"), d.k_pool,
        d.v_pool, d.tables, torch.tensor([620], dtype=torch.int32, device="cuda"), 120, 0, w.scale)
    second = pkv.paged_prefill_chunk_attention(
        d.q[120:].contiguous(), torch.tensor([0, 80], dtype=torch.int32, device="cuda"), d.k_pool,
        d.v_pool, d.tables, d.seq_lens, 80, 0, w.scale)
    torch.cuda.synchronize()
    assert_close(to_f64(torch.cat([first, second])), to_f64(one), "bf16", "two chunks vs one")


def test_deterministic(pkv):
    w = gen.prefill_workload(seed=72, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                             prefix_lens=[2000, 700], chunk_lens=[300, 128])
    d = Dev(w)
    append(pkv, d)
    a = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 300,
                                          0, w.scale).clone()
    b = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 300,
                                          0, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and int(d.status.item()) == 0


def test_unsupported_shape_reported(pkv):
    # head_dim 64 runs only as a short chunk (on the decode kernel); 8 queries
    # x 3 heads per kv head do not fit its 16-row tile
    w = gen.prefill_workload(seed=73, dtype="bf16", num_q_heads=6, num_kv_heads=2, head_dim=64,
                             prefix_lens=[10], chunk_lens=[8])
    d = Dev(w)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 8, 0,
                                          w.scale)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("scale", [-0.3, 0.0, 0.5])
def test_scale_sign_and_zero(pkv, orc, scale):
    # a negative scale is staged as -q (exact), a zero scale attends uniformly
    import dataclasses
    w = gen.prefill_workload(seed=74, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                             prefix_lens=[0, 90, 300], chunk_lens=[37, 64, 130])
    w = dataclasses.replace(w, scale=scale)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "bf16", f"prefill scale {scale}")


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 1), (16, 16)])
@pytest.mark.parametrize("window", [0, 64])
def test_verify_steps(pkv, orc, hq, hkv, window):
    # speculative-verify shape: a few queries per row over a long paged
    # context; the chunk fits the first query tile, the second stays idle
    w = gen.prefill_workload(seed=80 + hq + hkv + window, dtype="bf16", num_q_heads=hq,
                             num_kv_heads=hkv, head_dim=128,
                             prefix_lens=[100, 1000, 3000, 17, 0], chunk_lens=[4, 4, 2, 8, 3],
                             window=window)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "bf16", f"verify {hq}/{hkv} w{window}")



@pytest.mark.parametrize("d,hq,hkv,chunks", [
    (128, 32, 8, [4, 4, 2, 1, 3]),    # 4 queries x 4 heads fill the 16-row tile
    (128, 16, 16, [8, 16, 1, 5, 9]),  # one head per kv head: up to 16 queries
    (64, 8, 2, [4, 2, 4, 1, 3]),
    (256, 8, 1, [2, 1, 2, 2, 1]),
    (128, 48, 16, [5, 1, 3, 5, 2]),   # 3 heads per kv head
])
@pytest.mark.parametrize("window", [0, 40])
def test_verify_steps_on_decode_kernel(pkv, orc, d, hq, hkv, chunks, window):
    # (query, head) pairs of a kv head within 16: the split-KV decode kernel
    # serves the chunk, one row of M per pair, causal within the chunk
    w = gen.prefill_workload(seed=90 + d + hq + window, dtype="bf16", num_q_heads=hq,
                             num_kv_heads=hkv, head_dim=d,
                             prefix_lens=[100, 1000, 3000, 17, 0], chunk_lens=chunks,
                             window=window)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "bf16", f"verify on decode d{d} {hq}/{hkv} w{window}")


# ---------------------------------------------------------------------------
# the persistent balanced schedule: more (row, kv head, query-tile pair)
# items than SMs; every CTA takes an equal share of the items' 64-key tiles,
# items cut by a CTA boundary are computed in pieces and merged
# ---------------------------------------------------------------------------

def _sk_on(pkv, w):
    """The call runs the balanced schedule (its workspace is the schedule's)."""
    import torch as _t
    C = int(np.max(np.diff(w.cu_q_lens)))
    G = w.num_q_heads // w.num_kv_heads
    items = w.batch * w.num_kv_heads * -(-C // (2 * (128 // G)))
    return items > _t.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("window", [0, 300])
def test_balanced_schedule_ragged(pkv, orc, window):
    # 8 ragged rows, 16 q / 4 kv heads: 320 items, short and long key ranges
    w = gen.prefill_workload(seed=75 + window, dtype="bf16", num_q_heads=16, num_kv_heads=4,
                             head_dim=128, prefix_lens=[0, 5, 130, 300, 1000, 17, 64, 2000],
                             chunk_lens=[600, 1, 64, 65, 300, 129, 512, 33], window=window)
    assert _sk_on(pkv, w)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "bf16", f"balanced schedule, window {window}")


def test_balanced_schedule_many_tiny_items(pkv, orc):
    # 40 rows of 70 queries with no prefix: items of one or two tiles, so a
    # CTA's share runs through many items and most boundaries cut one
    w = gen.prefill_workload(seed=77, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                             prefix_lens=[0] * 40, chunk_lens=[70] * 40)
    assert _sk_on(pkv, w)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "bf16", "balanced schedule, tiny items")


def test_balanced_schedule_items_just_past_sms(pkv, orc):
    # a few items more than SMs: each CTA runs one item whole, then the few
    # remaining items' tiles are shared by all CTAs, so each of them is cut
    # into about twenty pieces that one warp merges
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    rows = -(-(n_sm + 8) // 32)  # 8 kv heads x 4 query-tile pairs per row
    w = gen.prefill_workload(seed=79, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                             prefix_lens=[1500 - 37 * r for r in range(rows)], chunk_lens=[256] * rows)
    assert _sk_on(pkv, w)
    got, ref, _ = run_prefill(pkv, orc, w)
    assert_close(got, ref, "bf16", "balanced schedule, items just past the SMs")


def test_balanced_schedule_deterministic(pkv):
    w = gen.prefill_workload(seed=78, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                             prefix_lens=[3000, 700, 50, 1200], chunk_lens=[512, 300, 600, 77])
    assert _sk_on(pkv, w)
    d = Dev(w)
    append(pkv, d)
    a = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 600,
                                          0, w.scale).clone()
    b = pkv.paged_prefill_chunk_attention(d.q, d.cu, d.k_pool, d.v_pool, d.tables, d.seq_lens, 600,
                                          0, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and int(d.status.item()) == 0
