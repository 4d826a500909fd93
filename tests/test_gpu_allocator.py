"""The host block allocator drives the GPU path: requests whose prompts share
leading blocks get tables from the allocator (shared ids for the shared full
blocks), the new tokens are appended through its slots, and decode - with and
without the shared-prefix read-once path - matches the oracle on those
tables.
"""
import dataclasses

import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import Dev, append, assert_close, oracle_pools, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


def test_allocator_tables_decode_matches_oracle(pkv, orc):
    bs, pool = 16, 512
    a = pkv.BlockAllocator(bs, 64, pool)
    system = list(range(1000, 1000 + 320))          # 20 full blocks shared by rows 0..3
    other = list(range(5000, 5000 + 50))
    prompts = [system + [1] * 37, system + [2] * 300, system + [3] * 5, system,
               other + [4] * 200]
    reqs, lens = [], []
    for p in prompts:
        r = a.begin()
        a.find_cached_prefix(r, p)
        a.reserve(r, len(p) + 1)                    # room for the decode step's token
        a.publish(r, p)
        reqs.append(r)
        lens.append(len(p))
    width = max(len(a.table(r)) for r in reqs)
    tables = np.full((len(reqs), width), -1, dtype=np.int32)
    for i, r in enumerate(reqs):
        t = a.table(r)
        tables[i, :len(t)] = t
    assert all((tables[i, :20] == tables[0, :20]).all() for i in range(4))
    assert a.stats()[0] <= pool

    w = gen.decode_workload(seed=90, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                            context_lens=lens, pool_blocks=pool, table_width=width, poison=False)
    w = dataclasses.replace(w, block_tables=tables)
    d = Dev(w)
    slots = append(pkv, d)
    or_slots, kp, vp = oracle_pools(orc, w)
    assert np.array_equal(slots, or_slots)
    ref = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    plain = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                       status=d.status)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, bs, d.k_pool.device)
    assert desc is not None and desc.num_groups >= 1
    shared = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0,
                                        w.scale, prefix=desc, status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert_close(to_f64(plain), ref, "bf16", "allocator tables, split path")
    assert_close(to_f64(shared), ref, "bf16", "allocator tables, shared-prefix path")


def test_sliding_group_with_expired_blocks(pkv, orc):
    # a sliding-window group: the allocator drops the blocks the window has
    # left (-1 sentinels in the tables) and decode reads only live blocks
    bs, pool, W = 16, 256, 64
    a = pkv.BlockAllocator(bs, 32, pool)
    prompts = [list(range(500)), list(range(1000, 1333)), list(range(40)), list(range(2000, 2100))]
    reqs, lens = [], []
    for p in prompts:
        r = a.begin()
        a.find_cached_prefix(r, p)
        a.reserve(r, len(p) + 1)
        a.publish(r, p)
        a.expire(r, max(0, len(p) + 1 - W))        # the window after this step's token
        reqs.append(r)
        lens.append(len(p))
    width = max(len(a.table(r)) for r in reqs)
    tables = np.full((len(reqs), width), -1, dtype=np.int32)
    for i, r in enumerate(reqs):
        t = a.table(r)
        tables[i, :len(t)] = t
    assert (tables[0, :27] == -1).all() and (tables[0, 27:] >= 0).all()   # 501 - 64 = 437 -> 27 blocks gone
    w = gen.decode_workload(seed=91, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=lens, window=W, pool_blocks=pool, table_width=width,
                            poison=False)
    w = dataclasses.replace(w, block_tables=tables)
    d = Dev(w)
    slots = append(pkv, d)
    or_slots, kp, vp = oracle_pools(orc, w)
    assert np.array_equal(slots, or_slots)
    ref = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, W, w.scale)
    got = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, W, w.scale,
                                     status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert_close(to_f64(got), ref, "bf16", "sliding group with expired blocks")
