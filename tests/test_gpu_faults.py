"""Faults only the device can see are reported in the status word, never by
a GPU fault: a bad block id, a slot past the pool, a length past the table,
a lying prefix descriptor.  Every injected fault is made on the host (a bad
value in an index array); each kernel bounds-checks before it reads."""
import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import Dev, append

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bad_block_id_sets_status(pkv, dtype):
    w = gen.decode_workload(seed=20, dtype=dtype, num_q_heads=4, num_kv_heads=2, head_dim=64,
                            context_lens=[100, 100])
    d = Dev(w)
    append(pkv, d)
    d.tables[0, 2] = w.num_blocks + 5
    d.tables[0, 3] = -7
    out = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                     status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) & pkv.DEV_BAD_BLOCK
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bad_slot_sets_status(pkv, dtype):
    w = gen.decode_workload(seed=21, dtype=dtype, num_q_heads=4, num_kv_heads=2, head_dim=64,
                            context_lens=[10, 20])
    d = Dev(w)
    before = d.k_pool.clone()
    slots = torch.tensor([w.num_blocks * 16 + 3, -1], dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(d.k_pool, d.v_pool, slots, d.k_new, d.v_new, status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == pkv.DEV_BAD_SLOT
    assert torch.equal(before.view(torch.uint8), d.k_pool.view(torch.uint8))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_length_past_table_sets_status(pkv, dtype):
    w = gen.decode_workload(seed=22, dtype=dtype, num_q_heads=4, num_kv_heads=2, head_dim=64,
                            context_lens=[30, 60])
    d = Dev(w)
    append(pkv, d)
    d.seq_lens[1] = 10_000
    d.seq_lens[0] = -5
    out = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                     status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) & pkv.DEV_BAD_LEN
    assert torch.all(out[0] == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lying_prefix_descriptor_sets_status(pkv, dtype):
    w = gen.decode_workload(seed=23, dtype=dtype, num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[64, 70, 90], shared_prefix_tokens=64)
    d = Dev(w)
    append(pkv, d)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, d.k_pool.device)
    # row 2 claims the prefix but holds other blocks there
    d.tables[2, 1] = int(w.block_tables[2, 4]) if w.block_tables.shape[1] > 4 else 0
    pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                               prefix=desc, status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) & pkv.DEV_BAD_PREFIX


def test_host_errors(pkv):
    w = gen.decode_workload(seed=24, dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=128,
                            context_lens=[30])
    d = Dev(w)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                   workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == pkv.PKV_ERR_WORKSPACE
    desc = pkv.PrefixDesc(1, 1, 1, torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.ones(1, dtype=torch.int32, device="cuda"))
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 16, w.scale,
                                   prefix=desc)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED


def test_buffers_off_the_gpu_rejected_before_launch(pkv):
    # a host tensor's pointer handed to a kernel would be dereferenced on the
    # device: the binding refuses such buffers before anything is enqueued
    w = gen.decode_workload(seed=25, dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=128,
                            context_lens=[30])
    d = Dev(w)
    n0 = pkv.launch_count()
    for kw in ({"workspace": torch.empty(1 << 20, dtype=torch.uint8)},
               {"out": torch.empty(tuple(d.q.shape), dtype=d.q.dtype)},
               {"status": torch.zeros(1, dtype=torch.int32)},
               {"status": torch.zeros(1, dtype=torch.int64, device="cuda")}):
        with pytest.raises(ValueError):
            pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                       **kw)
    slots = torch.zeros(w.k_new.shape[0], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        pkv.paged_kv_append(d.k_pool, d.v_pool, slots, d.k_new.cpu(), d.v_new)
    with pytest.raises(ValueError):
        pkv.paged_decode_attention_no_alloc(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0,
                                            w.scale, torch.empty(tuple(d.q.shape), dtype=d.q.dtype))
    assert pkv.launch_count() == n0
