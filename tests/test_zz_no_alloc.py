"""The allocation-free decode entry point (GPU; this file is collected last).

paged_decode_attention_no_alloc serves callers that cannot allocate device
memory where they call the library (a plug-in inside a framework that owns all
device memory, a serving loop that bans cudaMalloc on its hot path): it takes
its scratch from a fixed array in the library's device image instead of a
workspace.  Here it must give what the workspace entry point gives, call after
call, and refuse sizes whose scratch would not fit.
"""
import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import Dev, append, assert_close, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


@pytest.mark.parametrize("dtype,prefix", [("bf16", True), ("bf16", False), ("f32", True)])
def test_no_alloc_matches_workspace_entry_point(pkv, dtype, prefix):
    suf = [int(x) for x in gen.uniform_ints(81, "s", 12, 0, 2000)]
    w = gen.decode_workload(seed=81, dtype=dtype, num_q_heads=16, num_kv_heads=4, head_dim=128,
                            context_lens=[256 + s for s in suf], shared_prefix_tokens=256)
    d = Dev(w)
    append(pkv, d)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, d.k_pool.device) if prefix else None
    ml = int(w.seq_lens.max())
    ref = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                     max_seq_len=ml, prefix=desc, status=d.status)
    torch.cuda.synchronize()
    ref = to_f64(ref)
    for call in range(2):  # two calls in a row share the scratch
        out = torch.full_like(d.q, float("nan"))
        pkv.paged_decode_attention_no_alloc(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0,
                                            w.scale, out, max_seq_len=ml, prefix=desc,
                                            status=d.status)
        torch.cuda.synchronize()
        assert int(d.status.item()) == 0
        assert_close(to_f64(out), ref, dtype, f"no-alloc call {call + 1}")


def test_no_alloc_rejects_requests_beyond_the_scratch(pkv):
    # 512 rows x 64 q heads: even one split per row needs 512 * 64 * 130 * 4
    # bytes of partials, more than the static scratch holds
    B, hq, hkv, D, width = 512, 64, 8, 128, 64
    need = pkv.decode_workspace_size(B, hq, hkv, D, 16, width * 16)
    assert need > pkv.NO_ALLOC_SCRATCH_BYTES
    kp = torch.zeros((1, hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((B, hq, D), dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros((B, width), dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_no_alloc(q, kp, kp, tables, lens, 0, 1.0, out)
    assert e.value.code == pkv.PKV_ERR_WORKSPACE
