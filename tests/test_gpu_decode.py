"""GPU parity of append + paged decode against the oracle (through the C ABI).

Tolerances: bf16 K/V with fp32 accumulation |gpu - ref| <= 2e-3 + 1e-2 |ref|;
f32 pools 1e-5 + 1e-5 |ref|; pools after the append and slot mappings bit-exact.
"""
import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import (Dev, append, assert_appended_blocks_equal, assert_close, oracle_pools,
                      sample_pairs, storage_bytes, to_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


def run_step(pkv, orc, w, prefix=False, pairs=None, check_pool=True):
    """Append + decode on the GPU; the oracle's output (full or sampled)."""
    d = Dev(w)
    slots = append(pkv, d)
    or_slots, kp, vp = oracle_pools(orc, w)
    assert np.array_equal(slots, or_slots)
    if check_pool:
        assert storage_bytes(d.k_pool) == kp.tobytes() and storage_bytes(d.v_pool) == vp.tobytes()
    else:
        assert_appended_blocks_equal(d, slots, kp, vp)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, w.block_size, d.k_pool.device) \
        if prefix else None
    out = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, w.window,
                                     w.scale, max_seq_len=int(w.seq_lens.max()), prefix=desc,
                                     status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    got = to_f64(out)
    if pairs is None:
        ref = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window, w.scale)
        return got, ref, d
    ref = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window, w.scale,
                     pairs=pairs)
    return got[pairs[:, 0], pairs[:, 1]], ref, d


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("prefix", [False, True])
def test_tiny_f32(pkv, orc, prefix):
    w = gen.tiny_f32()
    got, ref, _ = run_step(pkv, orc, w, prefix=prefix)
    assert_close(got, ref, "f32", "tiny f32")


def test_dense_bf16(pkv, orc):
    w = gen.dense_bf16()
    got, ref, _ = run_step(pkv, orc, w)
    assert_close(got, ref, "bf16", "dense bf16")


@pytest.mark.parametrize("prefix", [False, True])
def test_shared_prefix_b32_full_size(pkv, orc, prefix):
    # every output element of the batch-32 step; the pools' appended blocks
    # byte for byte (the whole pools are too large to copy back)
    w = gen.shared_prefix_b32()
    got, ref, _ = run_step(pkv, orc, w, prefix=prefix, check_pool=False)
    assert got.shape == ref.shape == (w.batch, w.num_q_heads, w.head_dim)
    assert_close(got, ref, "bf16", f"shared prefix b32 (prefix path {prefix})")


def test_long_two_groups_full_size(pkv, orc):
    # both groups of the long-context workload, every output element
    full, sliding = gen.long_two_groups()
    for w in (full, sliding):
        got, ref, _ = run_step(pkv, orc, w, check_pool=False)
        assert got.shape == ref.shape == (w.batch, w.num_q_heads, w.head_dim)
        assert_close(got, ref, "bf16", w.name)


# ---------------------------------------------------------------------------
# shapes, windows, ragged lengths (small enough for the full oracle)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,hq,hkv", [(64, 4, 4), (128, 8, 2), (128, 32, 8), (256, 8, 1),
                                      (64, 16, 1), (128, 6, 2)])
@pytest.mark.parametrize("window", [0, 1, 37, 200])
def test_shapes_windows_ragged(pkv, orc, dtype, d, hq, hkv, window):
    ctx = [0, 1, 15, 16, 17, 100, 333, 700]
    w = gen.decode_workload(seed=100 + d + hq + window, dtype=dtype, num_q_heads=hq,
                            num_kv_heads=hkv, head_dim=d, context_lens=ctx, window=window)
    got, ref, _ = run_step(pkv, orc, w)
    assert_close(got, ref, dtype, f"{dtype} d{d} {hq}/{hkv} w{window}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_scale_sign_and_zero(pkv, orc, dtype, scale):
    import dataclasses
    w = gen.decode_workload(seed=9, dtype=dtype, num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[1, 30, 300, 1000])
    w = dataclasses.replace(w, scale=scale)
    got, ref, _ = run_step(pkv, orc, w)
    assert_close(got, ref, dtype, f"{dtype} decode scale {scale}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sliding_null_sentinel(pkv, orc, dtype):
    w = gen.decode_workload(seed=7, dtype=dtype, num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[40, 500, 1000, 63], window=48, sliding_live_only=True)
    assert (w.block_tables < 0).any()
    got, ref, _ = run_step(pkv, orc, w)
    assert_close(got, ref, dtype, "sliding with null sentinel")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefix_groups_mixed(pkv, orc, dtype):
    # rows 0..5 share a 5-block prefix; other rows private; lengths ragged
    w = gen.decode_workload(seed=8, dtype=dtype, num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[80, 81, 95, 96, 300, 1000], shared_prefix_tokens=80)
    got, ref, _ = run_step(pkv, orc, w, prefix=True)
    assert_close(got, ref, dtype, "prefix path")
    got2, _, _ = run_step(pkv, orc, w, prefix=False)
    assert_close(got2, ref, dtype, "no prefix path")


def test_prefix_with_window_is_refused(pkv, orc):
    # the shared-prefix path serves full attention only: a window with a
    # prefix descriptor is refused before any launch, the output untouched
    w = gen.decode_workload(seed=8, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[80, 81, 95, 96, 300, 1000], shared_prefix_tokens=80)
    d = Dev(w)
    append(pkv, d)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, w.block_size, d.k_pool.device)
    out = torch.full_like(d.q, 7.0)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 64, w.scale,
                                   max_seq_len=int(w.seq_lens.max()), prefix=desc, out=out,
                                   status=d.status)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and int(d.status.item()) == 0


def test_prefix_many_rows_two_chunks(pkv, orc):
    # 40 rows x 4 heads = 160 pairs: two row chunks of the prefix CTAs
    suf = [int(x) for x in gen.uniform_ints(9, "s", 40, 0, 300)]
    w = gen.decode_workload(seed=9, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                            context_lens=[160 + s for s in suf], shared_prefix_tokens=160)
    got, ref, _ = run_step(pkv, orc, w, prefix=True)
    assert_close(got, ref, "bf16", "prefix two chunks")


def test_empty_rows_give_zeros(pkv):
    w = gen.decode_workload(seed=10, dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=128,
                            context_lens=[5, 20])
    d = Dev(w)
    append(pkv, d)
    d.seq_lens[0] = 0
    out = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                     status=d.status)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0) and torch.isfinite(out[1].float()).all()
    assert int(d.status.item()) == 0


# ---------------------------------------------------------------------------
# invariances the pages state (bit-exact on the GPU)
# ---------------------------------------------------------------------------

def _decode(pkv, d, w, window=None, prefix=None, max_seq_len=None):
    out = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens,
                                     w.window if window is None else window, w.scale,
                                     prefix=prefix, max_seq_len=max_seq_len, status=d.status)
    torch.cuda.synchronize()
    return out.clone()


def test_run_to_run_deterministic(pkv):
    w = gen.decode_workload(seed=11, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                            context_lens=[3000, 17, 2048, 999])
    d = Dev(w)
    append(pkv, d)
    a, b = _decode(pkv, d, w), _decode(pkv, d, w)
    assert torch.equal(a, b)


def test_over_split_gives_same_bits(pkv):
    # any split size at or above a row's block count is one split: same bits
    w = gen.decode_workload(seed=12, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                            context_lens=[300, 511, 40])
    d = Dev(w)
    append(pkv, d)
    try:
        pkv.set_decode_split_blocks(32)
        a = _decode(pkv, d, w)
        pkv.set_decode_split_blocks(64)
        b = _decode(pkv, d, w)
        pkv.set_decode_split_blocks(4)
        c = _decode(pkv, d, w)
    finally:
        pkv.set_decode_split_blocks(0)
    assert torch.equal(a, b)
    assert_close(to_f64(c), to_f64(a), "bf16", "split 4 vs 32")


def test_batched_equals_per_row(pkv):
    w = gen.decode_workload(seed=13, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[100, 900, 33, 2000])
    d = Dev(w)
    append(pkv, d)
    try:
        pkv.set_decode_split_blocks(16)
        full = _decode(pkv, d, w)
        for r in range(w.batch):
            q = d.q[r:r + 1].contiguous()
            out = pkv.paged_decode_attention(q, d.k_pool, d.v_pool, d.tables[r:r + 1].contiguous(),
                                             d.seq_lens[r:r + 1].contiguous(), 0, w.scale)
            torch.cuda.synchronize()
            assert torch.equal(out[0], full[r]), r
    finally:
        pkv.set_decode_split_blocks(0)


def test_block_relabelling_invariant(pkv):
    w = gen.decode_workload(seed=14, dtype="bf16", num_q_heads=8, num_kv_heads=4, head_dim=64,
                            context_lens=[77, 400, 1023])
    d = Dev(w)
    append(pkv, d)
    a = _decode(pkv, d, w)
    perm = torch.from_numpy(gen.permutation(5, "relabel", w.num_blocks)).cuda()
    k2, v2 = torch.empty_like(d.k_pool), torch.empty_like(d.v_pool)
    k2[perm], v2[perm] = d.k_pool, d.v_pool
    d.k_pool, d.v_pool = k2, v2
    d.tables = torch.where(d.tables >= 0, perm[d.tables.clamp(min=0).long()].int(), d.tables)
    b = _decode(pkv, d, w)
    assert torch.equal(a, b)


def test_row_isolation(pkv):
    w = gen.decode_workload(seed=15, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[200, 300, 400])
    d = Dev(w)
    append(pkv, d)
    a = _decode(pkv, d, w)
    # change row 1's query and its private blocks
    d.q[1] = -d.q[1]
    blk = d.tables[1][d.tables[1] >= 0].long()
    d.k_pool[blk] = d.k_pool[blk] * 2
    b = _decode(pkv, d, w)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2]) and not torch.equal(a[1], b[1])


def test_shared_equals_private_copies(pkv, orc):
    w = gen.decode_workload(seed=16, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                            context_lens=[256, 300, 1000, 256], shared_prefix_tokens=256)
    d = Dev(w)
    append(pkv, d)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, d.k_pool.device)
    assert desc is not None and desc.num_groups == 1
    shared_on = _decode(pkv, d, w, prefix=desc)
    shared_off = _decode(pkv, d, w)
    # private copies of the prefix blocks for rows 1..3
    P = 16
    nb = w.num_blocks
    k2 = torch.cat([d.k_pool, torch.empty((3 * P,) + d.k_pool.shape[1:], dtype=d.k_pool.dtype,
                                          device="cuda")])
    v2 = torch.cat([d.v_pool, torch.empty_like(k2[nb:])])
    t2 = d.tables.clone()
    for r in range(1, 4):
        for j in range(P):
            new = nb + (r - 1) * P + j
            k2[new], v2[new] = d.k_pool[t2[r, j]], d.v_pool[t2[r, j]]
            t2[r, j] = new
    d2 = Dev(w)
    d2.q, d2.k_pool, d2.v_pool, d2.tables, d2.seq_lens = d.q, k2, v2, t2, d.seq_lens
    private = _decode(pkv, d2, w)
    assert torch.equal(private, shared_off)  # the same blocks, relabelled
    assert_close(to_f64(shared_on), to_f64(private), "bf16", "read-once prefix vs private copies")


@pytest.mark.parametrize("d,hq,hkv", [(64, 8, 2), (128, 32, 8), (256, 8, 1)])
def test_repeated_calls_stable_across_split_sizes(pkv, d, hq, hkv):
    # every split size gives a clean status and the same bits call after call
    # (a pipeline that lets a consumer run a full ring ahead fails this)
    w = gen.decode_workload(seed=17, dtype="bf16", num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            context_lens=[4000, 1500, 30, 2900])
    d_ = Dev(w)
    append(pkv, d_)
    try:
        for C in (0, 4, 12, 20, 40, 100, 300):
            pkv.set_decode_split_blocks(C)
            ref = _decode(pkv, d_, w)
            for _ in range(10):
                out = _decode(pkv, d_, w)
                assert torch.equal(out, ref), C
            assert int(d_.status.item()) == 0, C
    finally:
        pkv.set_decode_split_blocks(0)
