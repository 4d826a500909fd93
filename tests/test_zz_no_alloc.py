"""The allocation-free decode entry point (GPU; this file is collected last).

paged_decode_attention_no_alloc serves callers that cannot allocate device
memory where they call the library (a plug-in inside a framework that owns all
device memory, a serving loop that bans cudaMalloc on its hot path): it takes
its scratch from a fixed array in the library's device image instead of a
workspace.  It makes the same split plan as the workspace entry point, so it
must give the same bits, call after call, match the oracle within the decode
tolerance, and refuse sizes whose scratch would not fit.
"""
import pytest

import pkv_inputs as gen
from gpu_util import Dev, append, assert_close, oracle_pools, to_f64, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KS, VS = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


def _workload(dtype):
    suf = [int(x) for x in gen.uniform_ints(81, "s", 12, 0, 2000)]
    return gen.decode_workload(seed=81, dtype=dtype, num_q_heads=16, num_kv_heads=4, head_dim=128,
                               context_lens=[256 + s for s in suf], shared_prefix_tokens=256)


def _check_two_calls(pkv, q, kp, vp, tables, lens, w, status, desc, ref_ws, ref_oracle, dtype,
                     scales=None):
    ml = int(w.seq_lens.max())
    kw = {} if scales is None else {"k_scale": scales[0], "v_scale": scales[1]}
    for call in range(2):  # two calls in a row share the scratch
        out = torch.full_like(q, float("nan"))
        pkv.paged_decode_attention_no_alloc(q, kp, vp, tables, lens, 0, w.scale, out,
                                            max_seq_len=ml, prefix=desc, status=status, **kw)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref_ws), f"no-alloc call {call + 1} differs from the workspace call"
        assert_close(to_f64(out), ref_oracle, dtype, f"no-alloc call {call + 1} vs the oracle")


@pytest.mark.parametrize("dtype,prefix", [("bf16", True), ("bf16", False), ("f32", True)])
def test_no_alloc_matches_workspace_entry_point(pkv, orc, dtype, prefix):
    w = _workload(dtype)
    d = Dev(w)
    append(pkv, d)
    _, kp, vp = oracle_pools(orc, w)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, d.k_pool.device) if prefix else None
    ml = int(w.seq_lens.max())
    ref = pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale,
                                     max_seq_len=ml, prefix=desc, status=d.status)
    torch.cuda.synchronize()
    ref_oracle = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    _check_two_calls(pkv, d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, w, d.status, desc, ref,
                     ref_oracle, dtype)


@pytest.mark.parametrize("prefix", [True, False])
def test_no_alloc_fp8_pools(pkv, orc, prefix):
    # FP8 (E4M3) pools filled by appending the workload's context and new rows
    # on both sides with the same per-layer scales
    w = _workload("bf16")
    dev = torch.device("cuda")
    kp_h, vp_h = gen.fp8_empty_pools(w)
    kp, vp = torch.from_numpy(kp_h).to(dev), torch.from_numpy(vp_h).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ctx = gen.live_slots(w)
    new_slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
    for s, kr, vr in (ctx, (new_slots, w.k_new, w.v_new)):
        pkv.paged_kv_append(kp, vp, torch.from_numpy(s).to(dev), to_torch(kr, "bf16"),
                            to_torch(vr, "bf16"), status=status, k_scale=KS, v_scale=VS)
        orc.append(kp_h, vp_h, "fp8", s, kr, vr, KS, VS)
    q = to_torch(w.q, "bf16")
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, dev) if prefix else None
    ref = pkv.paged_decode_attention(q, kp, vp, tables, lens, 0, w.scale,
                                     max_seq_len=int(w.seq_lens.max()), prefix=desc, status=status,
                                     k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_oracle = orc.decode(w.q, kp_h, vp_h, "fp8", w.block_tables, w.seq_lens, 0, w.scale,
                            k_scale=KS, v_scale=VS)
    _check_two_calls(pkv, q, kp, vp, tables, lens, w, status, desc, ref, ref_oracle, "bf16",
                     scales=(KS, VS))


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
