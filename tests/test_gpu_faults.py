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


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 64), ("bf16", 128), ("bf16", 256)])
def test_bad_block_id_sets_status(pkv, dtype, d):
    w = gen.decode_workload(seed=20, dtype=dtype, num_q_heads=4, num_kv_heads=2, head_dim=d,
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


# ---------------------------------------------------------------------------
# fail-closed drill: a pipeline wait that runs out.  The drill leaves every
# pipeline's first load unissued and shortens the data-wait limit to 1 ms, so
# the wait for that load runs out with nothing in flight on its barrier; the
# CTA then lets the copies it did issue land and exits.  The status word must
# carry PKV_DEV_TIMEOUT, the call must return, and the next call (drill off)
# must be clean and match the oracle.
# ---------------------------------------------------------------------------
DRILL_NS = 1_000_000


def _drill(pkv, fn):
    pkv.set_wait_drill(DRILL_NS, pkv.DRILL_WITHHOLD_FIRST_LOAD)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        pkv.set_wait_drill()


@pytest.mark.parametrize("prefix", [False, True])
def test_wait_timeout_drill_decode_bf16(pkv, orc, prefix):
    from gpu_util import assert_close, oracle_pools, to_f64
    w = gen.decode_workload(seed=25, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[300, 700, 64], shared_prefix_tokens=64 if prefix else 0)
    d = Dev(w)
    append(pkv, d)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, d.k_pool.device) if prefix else None

    def call():
        return pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                          prefix=desc, status=d.status)

    _drill(pkv, call)
    assert int(d.status.item()) & pkv.DEV_TIMEOUT
    d.status.zero_()
    out = call()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    _, kp, vp = oracle_pools(orc, w)
    ref = orc.decode(w.q, kp, vp, "bf16", w.block_tables, w.seq_lens, 0, w.scale)
    assert_close(to_f64(out), ref, "bf16", "decode after the drill")


def test_wait_timeout_drill_decode_fp8(pkv):
    w = gen.decode_workload(seed=26, dtype="bf16", num_q_heads=8, num_kv_heads=1, head_dim=256,
                            context_lens=[200, 900])
    d = Dev(w)
    kp, vp = pkv.fp8_pools(w.num_blocks, 1, 256, "cuda")
    slots, kr, vr = gen.live_slots(w)
    ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)
    from gpu_util import to_torch
    pkv.paged_kv_append(kp, vp, torch.from_numpy(slots).cuda(), to_torch(kr, "bf16"),
                        to_torch(vr, "bf16"), status=d.status, k_scale=ks, v_scale=vs)

    def call():
        return pkv.paged_decode_attention(d.q, kp, vp, d.tables, d.seq_lens, 0, w.scale,
                                          status=d.status, k_scale=ks, v_scale=vs)

    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    ref = call().clone()
    _drill(pkv, call)
    assert int(d.status.item()) & pkv.DEV_TIMEOUT
    d.status.zero_()
    out = call()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("fp8", [False, True])
def test_wait_timeout_drill_prefill(pkv, fp8):
    w = gen.prefill_workload(seed=27, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                             prefix_lens=[640, 100], chunk_lens=[200, 130])
    d = Dev(w)
    kw = {}
    if fp8:
        kp, vp = pkv.fp8_pools(w.num_blocks, 2, 128, "cuda")
        from gpu_util import to_torch
        ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)
        slots, kr, vr = gen.live_slots(w)
        pkv.paged_kv_append(kp, vp, torch.from_numpy(slots).cuda(), to_torch(kr, "bf16"),
                            to_torch(vr, "bf16"), status=d.status, k_scale=ks, v_scale=vs)
        kw = {"k_scale": ks, "v_scale": vs}
    else:
        kp, vp = d.k_pool, d.v_pool
    new = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows,
                                                 w.new_pos, 16)).cuda()
    pkv.paged_kv_append(kp, vp, new, d.k_new, d.v_new, status=d.status, **kw)
    C = int(np.max(np.diff(w.cu_q_lens)))

    def call():
        return pkv.paged_prefill_chunk_attention(d.q, d.cu, kp, vp, d.tables, d.seq_lens, C, 0,
                                                 w.scale, status=d.status, **kw)

    ref = call().clone()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    _drill(pkv, call)
    assert int(d.status.item()) & pkv.DEV_TIMEOUT
    d.status.zero_()
    out = call()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("fp8", [False, True])
def test_wait_timeout_drill_prefill_balanced_schedule(pkv, fp8):
    # more (row, kv head, query-tile pair) items than SMs: the persistent
    # balanced schedule, every CTA's first load withheld
    w = gen.prefill_workload(seed=28, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                             prefix_lens=[0] * 40, chunk_lens=[70] * 40)
    assert w.batch * w.num_kv_heads * 2 > torch.cuda.get_device_properties(0).multi_processor_count
    d = Dev(w)
    kw = {}
    if fp8:
        kp, vp = pkv.fp8_pools(w.num_blocks, 4, 128, "cuda")
        ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)
        kw = {"k_scale": ks, "v_scale": vs}
    else:
        kp, vp = d.k_pool, d.v_pool
    new = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows,
                                                 w.new_pos, 16)).cuda()
    pkv.paged_kv_append(kp, vp, new, d.k_new, d.v_new, status=d.status, **kw)

    def call():
        return pkv.paged_prefill_chunk_attention(d.q, d.cu, kp, vp, d.tables, d.seq_lens, 70, 0,
                                                 w.scale, status=d.status, **kw)

    ref = call().clone()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    _drill(pkv, call)
    assert int(d.status.item()) & pkv.DEV_TIMEOUT
    d.status.zero_()
    out = call()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert torch.equal(out, ref)


def test_wait_drill_rejects_unknown_flags(pkv):
    with pytest.raises(pkv.PkvError):
        pkv.set_wait_drill(0, 2)
