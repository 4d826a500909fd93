"""GPU append: the pools after paged_kv_append equal the oracle's byte for byte."""
import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import Dev, append, oracle_pools, storage_bytes

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


@pytest.mark.parametrize("dtype,d,hkv", [("f32", 32, 3), ("f32", 64, 2), ("bf16", 64, 1),
                                         ("bf16", 128, 8), ("bf16", 256, 1)])
def test_chunk_append_bit_exact(pkv, orc, dtype, d, hkv):
    w = gen.prefill_workload(seed=30 + d, dtype=dtype, num_q_heads=hkv, num_kv_heads=hkv,
                             head_dim=d, prefix_lens=[0, 13, 64, 250], chunk_lens=[5, 77, 16, 300])
    dv = Dev(w)
    slots = append(pkv, dv)
    or_slots, kp, vp = oracle_pools(orc, w)
    torch.cuda.synchronize()
    assert np.array_equal(slots, or_slots)
    assert storage_bytes(dv.k_pool) == kp.tobytes() and storage_bytes(dv.v_pool) == vp.tobytes()
    assert int(dv.status.item()) == 0


def test_chunked_prefill_workload_append(pkv, orc):
    w = gen.chunked_prefill()
    dv = Dev(w)
    append(pkv, dv)
    _, kp, vp = oracle_pools(orc, w)
    torch.cuda.synchronize()
    assert storage_bytes(dv.k_pool) == kp.tobytes() and storage_bytes(dv.v_pool) == vp.tobytes()


def test_negative_slots_skipped(pkv):
    w = gen.decode_workload(seed=31, dtype="bf16", num_q_heads=2, num_kv_heads=2, head_dim=128,
                            context_lens=[3, 4, 5])
    dv = Dev(w)
    before = storage_bytes(dv.k_pool)
    pkv.paged_kv_append(dv.k_pool, dv.v_pool, torch.full((3,), -1, dtype=torch.int32, device="cuda"),
                        dv.k_new, dv.v_new, status=dv.status)
    torch.cuda.synchronize()
    assert storage_bytes(dv.k_pool) == before and int(dv.status.item()) == 0
