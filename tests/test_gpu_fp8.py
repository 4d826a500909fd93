"""GPU parity of the FP8 (E4M3) KV pools against the oracle (through the C ABI).

The pools start as the poison code everywhere; the context of a workload is
written by appending its live rows (bf16) and then the step's new rows, on the
GPU by the library and on the CPU by the oracle, from the same arrays.  The
pool bytes must agree exactly (the code of every element is decided by the
same float32 quotient on both sides); attention outputs within the bf16
tolerance |gpu - ref| <= 2e-3 + 1e-2 |ref| (the oracle attends the exact code
values in float64).
"""
import dataclasses

import numpy as np
import pytest

import pkv_inputs as gen
from gpu_util import assert_close, oracle_decode_rows, to_f64, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KS, VS = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_paged_kv_gb300 as m
    return m


def _rows_only(w, rows):
    """live slots of the blocks that the given rows' tables reach"""
    s, kr, vr = gen.live_slots(w)
    t = w.block_tables[np.asarray(rows)]
    keep = np.isin(s // 16, t[t >= 0])
    return s[keep], kr[keep], vr[keep]


class Fp8Step:
    """One workload on FP8 pools: context + new rows appended on both sides."""

    def __init__(self, pkv, orc, w, rows=None, check_pool=True):
        assert w.dtype == "bf16"
        dev = torch.device("cuda")
        self.w = w
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        kp, vp = gen.fp8_empty_pools(w)
        self.k_pool = torch.from_numpy(kp).to(dev)
        self.v_pool = torch.from_numpy(vp).to(dev)
        ctx = gen.live_slots(w) if rows is None else _rows_only(w, rows)
        new_slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
        or_slots, bad = orc.slot_mapping(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
        assert bad == 0 and np.array_equal(new_slots, or_slots)
        for s, kr, vr in (ctx, (new_slots, w.k_new, w.v_new)):
            if s.shape[0] == 0:
                continue
            pkv.paged_kv_append(self.k_pool, self.v_pool, torch.from_numpy(s).to(dev),
                                to_torch(kr, "bf16"), to_torch(vr, "bf16"), status=self.status,
                                k_scale=KS, v_scale=VS)
            orc.append(kp, vp, "fp8", s, kr, vr, KS, VS)
        self.kp, self.vp = kp, vp
        self.q = to_torch(w.q, "bf16")
        self.tables = torch.from_numpy(w.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.cu = torch.from_numpy(w.cu_q_lens).to(dev) if w.cu_q_lens is not None else None
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        if check_pool:
            assert np.array_equal(self.k_pool.cpu().numpy(), kp), "K pool bytes differ"
            assert np.array_equal(self.v_pool.cpu().numpy(), vp), "V pool bytes differ"
        else:
            # the blocks that received the step's new tokens, byte for byte
            blocks = np.unique(new_slots[new_slots >= 0] // 16)
            idx = torch.from_numpy(blocks.astype(np.int64)).to(dev)
            assert np.array_equal(self.k_pool.index_select(0, idx).cpu().numpy(), kp[blocks])
            assert np.array_equal(self.v_pool.index_select(0, idx).cpu().numpy(), vp[blocks])

    def decode(self, pkv, prefix=False):
        w = self.w
        desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, self.k_pool.device) \
            if prefix else None
        out = pkv.paged_decode_attention(self.q, self.k_pool, self.v_pool, self.tables,
                                         self.seq_lens, w.window, w.scale,
                                         max_seq_len=int(w.seq_lens.max()), prefix=desc,
                                         status=self.status, k_scale=KS, v_scale=VS)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        return to_f64(out)

    def oracle_decode(self, orc, pairs=None):
        w = self.w
        return orc.decode(w.q, self.kp, self.vp, "fp8", w.block_tables, w.seq_lens, w.window,
                          w.scale, pairs=pairs, k_scale=KS, v_scale=VS)


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d,hkv", [(64, 1), (128, 8), (256, 2)])
def test_append_codes_bit_exact(pkv, orc, d, hkv):
    w = gen.decode_workload(seed=300 + d + hkv, dtype="bf16", num_q_heads=hkv * 2,
                            num_kv_heads=hkv, head_dim=d, context_lens=[0, 1, 15, 16, 17, 70, 333])
    Fp8Step(pkv, orc, w)


def test_append_saturates_and_keeps_tiny_values(pkv, orc):
    # rows scaled to reach past +-448 * scale and down into the subnormal codes,
    # with zeros of both signs
    w = gen.decode_workload(seed=310, dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=128,
                            context_lens=[40, 5])
    f = gen.bf16_to_f32(w.k_new)
    mags = np.array([1e3, 30.0, 1.0, 1e-4, 3e-6], np.float32)
    k = f * mags[np.arange(f.size) % mags.size].reshape(f.shape)
    k.reshape(-1)[:4] = [0.0, -0.0, 448 * KS * 1.0001, -1e30]
    w = dataclasses.replace(w, k_new=gen.bf16_bits(k), v_new=gen.bf16_bits(k[::-1].copy()))
    s = Fp8Step(pkv, orc, w)
    codes = s.k_pool.cpu().numpy()
    assert (codes == 0x7E).any() and (codes == 0xFE).any(), "saturated codes present"
    assert ((codes & 0x78) == 0).sum() > 0, "subnormal or zero codes present"


@pytest.mark.parametrize("d,hkv", [(64, 2), (128, 8), (256, 1)])
@pytest.mark.parametrize("shuffle", [False, True])
def test_append_chunks_whole_blocks_and_ragged_ends(pkv, orc, d, hkv, shuffle):
    # chunks that start mid-block: whole blocks inside (written as tiles when
    # their 16 tokens come in order) and ragged ends (written token by token);
    # shuffled, no block has its tokens in order
    w = gen.prefill_workload(seed=315 + d, dtype="bf16", num_q_heads=hkv, num_kv_heads=hkv,
                             head_dim=d, prefix_lens=[0, 13, 64, 250], chunk_lens=[5, 77, 16, 300])
    slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
    order = np.arange(slots.shape[0])
    if shuffle:
        order = gen.permutation(316, "order", slots.shape[0]).astype(np.int64)
    s, kr, vr = slots[order], w.k_new[order], w.v_new[order]
    kp, vp = gen.fp8_empty_pools(w)
    k_d, v_d = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(k_d, v_d, torch.from_numpy(np.ascontiguousarray(s)).cuda(),
                        to_torch(np.ascontiguousarray(kr), "bf16"),
                        to_torch(np.ascontiguousarray(vr), "bf16"), status=status,
                        k_scale=KS, v_scale=VS)
    orc.append(kp, vp, "fp8", np.ascontiguousarray(s), np.ascontiguousarray(kr),
               np.ascontiguousarray(vr), KS, VS)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(k_d.cpu().numpy(), kp) and np.array_equal(v_d.cpu().numpy(), vp)


@pytest.mark.parametrize("d,hkv", [(64, 8), (64, 9), (128, 8), (128, 3), (256, 2), (256, 5)])
@pytest.mark.parametrize("shuffle", [False, True])
def test_append_bulk_windows_bit_exact(pkv, orc, d, hkv, shuffle):
    # a bulk append (2000+ tokens, the windowed kernel: whole blocks as tiles
    # staged a few kv heads at a time, ragged chunk ends token by token; the
    # head counts leave partial staging rounds), every pool byte against the
    # oracle; shuffled, no block is whole
    w = gen.prefill_workload(seed=317 + d + hkv, dtype="bf16", num_q_heads=hkv, num_kv_heads=hkv,
                             head_dim=d, prefix_lens=[0, 13, 250, 7], chunk_lens=[700, 333, 500, 611])
    slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
    assert slots.shape[0] >= 2048
    order = np.arange(slots.shape[0])
    if shuffle:
        order = gen.permutation(318, "order", slots.shape[0]).astype(np.int64)
    s, kr, vr = (np.ascontiguousarray(a[order]) for a in (slots, w.k_new, w.v_new))
    kp, vp = gen.fp8_empty_pools(w)
    k_d, v_d = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(k_d, v_d, torch.from_numpy(s).cuda(), to_torch(kr, "bf16"),
                        to_torch(vr, "bf16"), status=status, k_scale=KS, v_scale=VS)
    orc.append(kp, vp, "fp8", s, kr, vr, KS, VS)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(k_d.cpu().numpy(), kp) and np.array_equal(v_d.cpu().numpy(), vp)


# a scale that puts 1.0 / scale 3 float32 ulps above the midpoint 1.0625
# between the E4M3 values 1.0 and 1.125 (and 2^k / scale above 1.0625 * 2^k)
_NEAR_TIE_SCALE = float(np.float32(1.0 / (1.0625 * (1 + 3 * 2.0 ** -24))))


# a scale at which x = 3 gives a quotient just above a midpoint that the
# plain product x * RN(1/s) would land on (the quantizer's correction step
# must restore the quotient's code)
_PRODUCT_ON_MIDPOINT_SCALE = 11.294116973876953


@pytest.mark.parametrize("bulk", [False, True])
@pytest.mark.parametrize("whole_blocks", [False, True])
@pytest.mark.parametrize("scale", [KS, 0.25, _NEAR_TIE_SCALE, _PRODUCT_ON_MIDPOINT_SCALE])
def test_append_codes_at_rounding_boundaries(pkv, orc, whole_blocks, scale, bulk):
    # rows whose quotients x / scale sit on and next to the midpoints between
    # neighbouring E4M3 values, both signs, normal and subnormal codes, 448:
    # with a power-of-two scale the quotients are exact ties; the crafted
    # scale puts powers of two a few ulps off a tie
    v = orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = np.concatenate([(v[:-1] + v[1:]) / 2, [448.0, 464.0]])
    b = gen.bf16_bits((mids * scale).astype(np.float32)).astype(np.int32)
    near = np.concatenate([b + k for k in (-2, -1, 0, 1, 2)] +
                          [gen.bf16_bits(np.float32(2.0) ** np.arange(-6, 8, dtype=np.float32))])
    near = near.astype(np.uint16)
    vals = np.concatenate([near, near | np.uint16(0x8000)])
    D, hkv = 128, 2
    T = 16 * (len(vals) // (D * hkv * 16) + 1)   # whole blocks of tokens
    if bulk:
        T = 2048  # the windowed bulk kernel
    kn = np.resize(vals, T * hkv * D).reshape(T, hkv, D).astype(np.uint16)
    vn = np.resize(vals[::-1], T * hkv * D).reshape(T, hkv, D).astype(np.uint16)
    if whole_blocks:
        slots = np.arange(16, 16 + T, dtype=np.int32)        # blocks 1.. in order
        nb = T // 16 + 1
    else:
        slots = np.arange(T, dtype=np.int32) * 16 + 3        # one token per block
        nb = T + 1
    shape = (nb, hkv, 16 * D)
    kp, vp = np.full(shape, 0x7F, np.uint8), np.full(shape, 0x7F, np.uint8)
    k_d, v_d = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
    pkv.paged_kv_append(k_d, v_d, torch.from_numpy(slots).cuda(), to_torch(kn, "bf16"),
                        to_torch(vn, "bf16"), k_scale=scale, v_scale=scale)
    orc.append(kp, vp, "fp8", slots, kn, vn, scale, scale)
    torch.cuda.synchronize()
    assert np.array_equal(k_d.cpu().numpy(), kp) and np.array_equal(v_d.cpu().numpy(), vp)


def test_append_negative_slots_skipped(pkv, orc):
    w = gen.decode_workload(seed=311, dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=64,
                            context_lens=[20, 40])
    dev = torch.device("cuda")
    k, v = pkv.fp8_pools(w.num_blocks, 2, 64, dev)
    before = k.clone()
    pkv.paged_kv_append(k, v, torch.full((2,), -1, dtype=torch.int32, device=dev),
                        to_torch(w.k_new, "bf16"), to_torch(w.v_new, "bf16"), k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert torch.equal(k, before)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d,hq,hkv", [(64, 4, 4), (128, 8, 2), (128, 32, 8), (256, 8, 1),
                                      (64, 16, 1), (128, 6, 2)])
@pytest.mark.parametrize("window", [0, 1, 37, 200])
def test_decode_shapes_windows_ragged(pkv, orc, d, hq, hkv, window):
    ctx = [0, 1, 15, 16, 17, 100, 333, 700]
    w = gen.decode_workload(seed=320 + d + hq + window, dtype="bf16", num_q_heads=hq,
                            num_kv_heads=hkv, head_dim=d, context_lens=ctx, window=window)
    s = Fp8Step(pkv, orc, w)
    assert_close(s.decode(pkv), s.oracle_decode(orc), "bf16", f"fp8 d{d} {hq}/{hkv} w{window}")


@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_decode_scale_sign_and_zero(pkv, orc, scale):
    w = gen.decode_workload(seed=330, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                            context_lens=[3, 90, 513])
    s = Fp8Step(pkv, orc, dataclasses.replace(w, scale=scale))
    assert_close(s.decode(pkv), s.oracle_decode(orc), "bf16", f"fp8 scale {scale}")


@pytest.mark.parametrize("prefix", [False, True])
def test_decode_shared_prefix(pkv, orc, prefix):
    w = gen.decode_workload(seed=340, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                            context_lens=[256 + x for x in (0, 5, 17, 300, 1000, 64)],
                            shared_prefix_tokens=256)
    s = Fp8Step(pkv, orc, w)
    assert_close(s.decode(pkv, prefix=prefix), s.oracle_decode(orc), "bf16",
                 f"fp8 shared prefix (prefix path {prefix})")


def test_decode_sliding_null_sentinel(pkv, orc):
    w = gen.decode_workload(seed=350, dtype="bf16", num_q_heads=8, num_kv_heads=1, head_dim=256,
                            context_lens=[600, 1000, 50], window=128, sliding_live_only=True)
    s = Fp8Step(pkv, orc, w)
    assert_close(s.decode(pkv), s.oracle_decode(orc), "bf16", "fp8 sliding group")


def test_decode_shared_prefix_b32_full_size(pkv, orc):
    # the shared-prefix batch at full size on FP8 pools, every output element
    # of every row, both prefix paths
    w = gen.shared_prefix_b32()
    s = Fp8Step(pkv, orc, w, check_pool=False)
    ref = oracle_decode_rows(orc, w.q, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, w.window,
                             w.scale, w.num_q_heads, k_scale=KS, v_scale=VS)
    for prefix in (False, True):
        got = s.decode(pkv, prefix=prefix)
        assert got.shape == ref.shape
        assert_close(got, ref, "bf16", f"fp8 shared prefix b32 (prefix path {prefix})")


def test_query_out_of_f16_range_flagged(pkv, orc):
    w = gen.decode_workload(seed=360, dtype="bf16", num_q_heads=4, num_kv_heads=1, head_dim=64,
                            context_lens=[30])
    s = Fp8Step(pkv, orc, w)
    q = s.q.clone()
    q[0, 2, 5] = 1e5
    pkv.paged_decode_attention(q, s.k_pool, s.v_pool, s.tables, s.seq_lens, 0, w.scale,
                               status=s.status, k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert int(s.status.item()) == pkv.DEV_Q_RANGE


# ---------------------------------------------------------------------------
# verify steps (a few queries per row) and longer chunks (tensor-core prefill)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d,hq,hkv,chunks", [
    (128, 32, 8, [4, 4, 2, 1, 3]),
    (64, 8, 2, [4, 2, 4, 1, 3]),
    (256, 8, 1, [2, 1, 2, 2, 1]),
])
@pytest.mark.parametrize("window", [0, 40])
def test_verify_steps(pkv, orc, d, hq, hkv, chunks, window):
    w = gen.prefill_workload(seed=370 + d + hq + window, dtype="bf16", num_q_heads=hq,
                             num_kv_heads=hkv, head_dim=d,
                             prefix_lens=[100, 1000, 3000, 17, 0], chunk_lens=chunks,
                             window=window)
    s = Fp8Step(pkv, orc, w)
    out = pkv.paged_prefill_chunk_attention(s.q, s.cu, s.k_pool, s.v_pool, s.tables, s.seq_lens,
                                            max(chunks), window, w.scale, status=s.status,
                                            k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert int(s.status.item()) == 0
    ref = orc.prefill(w.q, w.cu_q_lens, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, window,
                      w.scale, k_scale=KS, v_scale=VS)
    assert_close(to_f64(out), ref, "bf16", f"fp8 verify d{d} {hq}/{hkv} w{window}")


def _prefill(pkv, s, w, window):
    out = pkv.paged_prefill_chunk_attention(s.q, s.cu, s.k_pool, s.v_pool, s.tables, s.seq_lens,
                                            int(np.max(np.diff(w.cu_q_lens))), window, w.scale,
                                            status=s.status, k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert int(s.status.item()) == 0
    return to_f64(out)


@pytest.mark.parametrize("hq,hkv,window", [(8, 2, 0), (32, 8, 0), (16, 16, 64), (8, 1, 200)])
def test_prefill_chunks(pkv, orc, hq, hkv, window):
    # chunks past 16 (query, head) pairs run on the tensor-core prefill kernel,
    # its softmax warpgroups widening the E4M3 tiles to f16 in shared memory
    w = gen.prefill_workload(seed=390 + hq + window, dtype="bf16", num_q_heads=hq,
                             num_kv_heads=hkv, head_dim=128, prefix_lens=[0, 90, 300, 1000],
                             chunk_lens=[37, 64, 130, 300], window=window)
    s = Fp8Step(pkv, orc, w)
    ref = orc.prefill(w.q, w.cu_q_lens, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, window,
                      w.scale, k_scale=KS, v_scale=VS)
    assert_close(_prefill(pkv, s, w, window), ref, "bf16", f"fp8 prefill {hq}/{hkv} w{window}")


@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_prefill_scale_sign_and_zero(pkv, orc, scale):
    w = gen.prefill_workload(seed=395, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                             prefix_lens=[0, 90, 300], chunk_lens=[37, 64, 130])
    w = dataclasses.replace(w, scale=scale)
    s = Fp8Step(pkv, orc, w)
    ref = orc.prefill(w.q, w.cu_q_lens, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, 0, w.scale,
                      k_scale=KS, v_scale=VS)
    assert_close(_prefill(pkv, s, w, 0), ref, "bf16", f"fp8 prefill scale {scale}")


def test_prefill_balanced_schedule(pkv, orc):
    # more (row, kv head, query-tile pair) items than SMs: the persistent
    # balanced schedule with FP8 widening, ragged rows, a window
    w = gen.prefill_workload(seed=398, dtype="bf16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                             prefix_lens=[0, 5, 130, 300, 1000, 17, 64, 900],
                             chunk_lens=[600, 1, 64, 65, 300, 129, 512, 33], window=200)
    assert w.batch * w.num_kv_heads * 10 > torch.cuda.get_device_properties(0).multi_processor_count
    s = Fp8Step(pkv, orc, w)
    ref = orc.prefill(w.q, w.cu_q_lens, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, 200, w.scale,
                      k_scale=KS, v_scale=VS)
    assert_close(_prefill(pkv, s, w, 200), ref, "bf16", "fp8 prefill, balanced schedule")


def test_prefill_items_just_past_sms(pkv, orc):
    # a few items more than SMs on FP8 pools: one whole item per CTA, then
    # the few remaining items cut into many pieces merged in the kernel
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    rows = -(-(n_sm + 8) // 32)  # 8 kv heads x 4 query-tile pairs per row
    w = gen.prefill_workload(seed=399, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                             prefix_lens=[1500 - 41 * r for r in range(rows)], chunk_lens=[256] * rows)
    s = Fp8Step(pkv, orc, w)
    ref = orc.prefill(w.q, w.cu_q_lens, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, 0, w.scale,
                      k_scale=KS, v_scale=VS)
    assert_close(_prefill(pkv, s, w, 0), ref, "bf16", "fp8 prefill, items just past the SMs")


def test_prefill_full_size(pkv, orc):
    # the chunked-prefill workload (4 x 512 queries after 16384 cached tokens)
    # on FP8 pools, sampled outputs
    w = gen.chunked_prefill()
    s = Fp8Step(pkv, orc, w, check_pool=False)
    got = _prefill(pkv, s, w, 0)
    u = gen.uniform_ints(396, "samples", 3 * 64, 0, 1 << 30)
    samples = np.array([(int(u[3 * k]) % w.batch, int(u[3 * k + 1]) % 512, int(u[3 * k + 2]) % 32)
                        for k in range(64)] + [(r, 511, 0) for r in range(w.batch)], dtype=np.int32)
    ref = orc.prefill(w.q, w.cu_q_lens, s.kp, s.vp, "fp8", w.block_tables, w.seq_lens, 0, w.scale,
                      samples=samples, k_scale=KS, v_scale=VS)
    rows = w.cu_q_lens[samples[:, 0]] + samples[:, 1]
    assert_close(got[rows, samples[:, 2]], ref, "bf16", "fp8 chunked prefill full size")


def test_prefill_query_range_flagged(pkv, orc):
    w = gen.prefill_workload(seed=397, dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                             prefix_lens=[16], chunk_lens=[64])
    s = Fp8Step(pkv, orc, w, check_pool=False)
    s.q[3, 1, 7] = 1e5
    pkv.paged_prefill_chunk_attention(s.q, s.cu, s.k_pool, s.v_pool, s.tables, s.seq_lens, 64, 0,
                                      w.scale, status=s.status, k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert int(s.status.item()) == pkv.DEV_Q_RANGE
