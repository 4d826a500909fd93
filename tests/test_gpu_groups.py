"""Fused decode over several groups (a full-attention group and sliding
groups of the same batch): one split launch and one merge launch.  Each
group's output equals its own paged_decode_attention call bit for bit and the
oracle within the tolerance.
"""
import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import Dev, append, assert_close, oracle_pools, to_f64, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


def _groups(seed, hq, hkv, d, ctx, windows):
    """One workload per group over the same rows: window 0 is a full group,
    window W > 0 a sliding group whose expired blocks hold the sentinel."""
    ws = []
    for i, W in enumerate(windows):
        ws.append(gen.decode_workload(seed=seed + 17 * i, dtype="bf16", num_q_heads=hq,
                                      num_kv_heads=hkv, head_dim=d, context_lens=ctx, window=W,
                                      sliding_live_only=W > 0))
    return ws


def _single(pkv, d, w):
    return pkv.paged_decode_attention(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, w.window,
                                      w.scale, max_seq_len=int(w.seq_lens.max()), status=d.status)


@pytest.mark.parametrize("hq,hkv,d,windows", [
    (8, 1, 256, [0, 128]),          # the long-context pair's shape
    (32, 8, 128, [0, 64]),
    (16, 4, 64, [0, 32, 200, 0]),   # four groups
    (12, 12, 128, [500]),           # one group
])
def test_groups_equal_single_calls_and_oracle(pkv, orc, hq, hkv, d, windows):
    ctx = [0, 5, 130, 700, 2047, 3000]
    ws = _groups(400 + d + hq, hq, hkv, d, ctx, windows)
    devs = [Dev(w) for w in ws]
    refs = []
    for w, dv in zip(ws, devs):
        slots = append(pkv, dv)
        or_slots, kp, vp = oracle_pools(orc, w)
        assert np.array_equal(slots, or_slots)
        refs.append(orc.decode(w.q, kp, vp, "bf16", w.block_tables, w.seq_lens, w.window, w.scale))
    groups = [pkv.DecodeGroup(dv.q, dv.k_pool, dv.v_pool, dv.tables, dv.seq_lens, w.window, w.scale,
                              max_seq_len=int(w.seq_lens.max())) for w, dv in zip(ws, devs)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = pkv.paged_decode_attention_groups(groups, status=status)
    singles = [_single(pkv, dv, w) for w, dv in zip(ws, devs)]
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and all(int(dv.status.item()) == 0 for dv in devs)
    for i, (o, s1, ref) in enumerate(zip(outs, singles, refs)):
        assert torch.equal(o, s1), f"group {i}: fused != single call"
        assert_close(to_f64(o), ref, "bf16", f"group {i} (window {windows[i]})")


def test_fp8_groups(pkv, orc):
    ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)
    ws = _groups(450, 8, 2, 128, [3, 90, 513, 1500], [0, 100])
    groups, refs, singles_args = [], [], []
    for w in ws:
        kp, vp = gen.fp8_empty_pools(w)
        k_d, v_d = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
        ctx_s, kr, vr = gen.live_slots(w)
        new_s = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
        for s_, a, b in ((ctx_s, kr, vr), (new_s, w.k_new, w.v_new)):
            pkv.paged_kv_append(k_d, v_d, torch.from_numpy(s_).cuda(), to_torch(a, "bf16"),
                                to_torch(b, "bf16"), k_scale=ks, v_scale=vs)
            orc.append(kp, vp, "fp8", s_, a, b, ks, vs)
        q = to_torch(w.q, "bf16")
        t = torch.from_numpy(w.block_tables).cuda()
        sl = torch.from_numpy(w.seq_lens).cuda()
        groups.append(pkv.DecodeGroup(q, k_d, v_d, t, sl, w.window, w.scale, k_scale=ks, v_scale=vs))
        singles_args.append((q, k_d, v_d, t, sl, w))
        refs.append(orc.decode(w.q, kp, vp, "fp8", w.block_tables, w.seq_lens, w.window, w.scale,
                               k_scale=ks, v_scale=vs))
    outs = pkv.paged_decode_attention_groups(groups)
    singles = [pkv.paged_decode_attention(q, k, v, t, sl, w.window, w.scale, k_scale=ks, v_scale=vs)
               for q, k, v, t, sl, w in singles_args]
    torch.cuda.synchronize()
    for i, (o, s1, ref) in enumerate(zip(outs, singles, refs)):
        assert torch.equal(o, s1)
        assert_close(to_f64(o), ref, "bf16", f"fp8 group {i}")


def test_long_two_groups_full_size(pkv, orc):
    full, sliding = gen.long_two_groups()
    devs = [Dev(w) for w in (full, sliding)]
    for dv in devs:
        append(pkv, dv)
    groups = [pkv.DecodeGroup(dv.q, dv.k_pool, dv.v_pool, dv.tables, dv.seq_lens, w.window, w.scale,
                              max_seq_len=int(w.seq_lens.max())) for w, dv in zip((full, sliding), devs)]
    outs = pkv.paged_decode_attention_groups(groups)
    singles = [_single(pkv, dv, w) for w, dv in zip((full, sliding), devs)]
    torch.cuda.synchronize()
    for o, s1 in zip(outs, singles):
        assert torch.equal(o, s1)
    # every output element of both groups against the oracle
    for w, o in zip((full, sliding), outs):
        _, kp, vp = oracle_pools(orc, w)
        ref = orc.decode(w.q, kp, vp, "bf16", w.block_tables, w.seq_lens, w.window, w.scale)
        assert ref.shape == tuple(o.shape)
        assert_close(to_f64(o), ref, "bf16", w.name)


def test_groups_must_share_the_head_shape(pkv):
    a = gen.decode_workload(seed=460, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[10, 20])
    b = gen.decode_workload(seed=461, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=64,
                            context_lens=[10, 20])
    da, db = Dev(a), Dev(b)
    groups = [pkv.DecodeGroup(d.q, d.k_pool, d.v_pool, d.tables, d.seq_lens, 0, w.scale)
              for w, d in ((a, da), (b, db))]
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_groups(groups)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    f = gen.decode_workload(seed=462, dtype="f32", num_q_heads=4, num_kv_heads=2, head_dim=64,
                            context_lens=[10])
    df = Dev(f)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_groups([pkv.DecodeGroup(df.q, df.k_pool, df.v_pool, df.tables,
                                                           df.seq_lens, 0, f.scale)])
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED
