"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` takes an oracle instance and raises AssertionError on a
mismatch.  ``tests/test_oracle_pins.py`` runs them against the normal build,
and against builds with a planted mistake to show that each mistake is caught.

What pins what:
  * append            -> numpy fancy-index assignment with the pool layout
                         definition; untouched bytes compared whole.
  * slot mapping      -> a hand-worked table; the inverse relation checked
                         for every position of every row.
  * decode / prefill  -> a dense attention written with numpy/scipy over keys
                         gathered by numpy indexing (the pages' paged == flat
                         gate, "paged-cache.md" parity-gate section); a 50-digit
                         mpmath brute force on tiny inputs; closed forms
                         (one key, zero query, equal keys, window 1, window
                         >= length, one dominant key); shared blocks == private
                         copies; physical block relabelling.
  * E4M3 codec        -> the published format table's values, the grid's
                         spacing, round trips, worked ties and saturation, a
                         brute-force nearest search;
  * FP8 tile layout   -> the PTX ISA's m16n8k16 B-fragment table;
  * FP8 append/attend -> the codec on float32 quotients; dense attention on
                         pools dequantized through the fragment table;
  * prefix groups     -> the pages' worked full-block example (a 1400-token
                         prompt at block size 16 has full blocks up to 1392,
                         "paged-cache.md" GDN ladder section) and the defining
                         properties (common run, full blocks, maximality).
"""
from __future__ import annotations

import math

import numpy as np

import pkv_inputs as gen


# ---------------------------------------------------------------------------
# independent helpers (numpy / scipy; no oracle code)
# ---------------------------------------------------------------------------

def gather_row(pool_f64: np.ndarray, tables: np.ndarray, r: int, g: int, lo: int, hi: int,
               bs: int) -> np.ndarray:
    pos = np.arange(lo, hi)
    return pool_f64[tables[r, pos // bs], g, pos % bs, :]


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    from scipy.special import softmax
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1])
    w = softmax(scale * (K @ q))
    return w @ V


def f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return gen.as_f32(a, dtype).astype(np.float64)


def oracle_slots(orc, w):
    slots, bad = orc.slot_mapping(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                  w.block_size)
    assert bad == 0
    return slots


def appended(orc, w):
    """Copies of the pools after the oracle's append."""
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    orc.append(kp, vp, w.dtype, oracle_slots(orc, w), w.k_new, w.v_new)
    return kp, vp


def small_decode(seed=7, dtype="f32", hq=4, hkv=2, d=16, ctx=(5, 20, 33), prefix=0, window=0,
                 bs=4, live_only=False):
    return gen.decode_workload(seed=seed, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=d, context_lens=list(ctx), block_size=bs,
                               shared_prefix_tokens=prefix, window=window,
                               pool_blocks=None, sliding_live_only=live_only)


# ---------------------------------------------------------------------------
# append and slot mapping
# ---------------------------------------------------------------------------

def pin_slot_mapping_hand_worked(orc):
    # rows of 37 and 50 tokens sharing blocks 5, 9; block size 16
    tables = np.array([[5, 9, 2, -1], [5, 9, 7, 11]], dtype=np.int32)
    rows = np.array([0, 1, 1, 0, 1], dtype=np.int32)
    pos = np.array([36, 49, 0, 15, 33], dtype=np.int32)
    slots, bad = orc.slot_mapping(tables, 12, rows, pos, 16)
    assert bad == 0
    assert slots.tolist() == [2 * 16 + 4, 11 * 16 + 1, 5 * 16, 5 * 16 + 15, 7 * 16 + 1]
    # a position past the table, and a sentinel entry, give -1
    slots, bad = orc.slot_mapping(tables, 12, np.array([0, 0], np.int32),
                                  np.array([48, 64], np.int32), 16)
    assert bad == 2 and slots.tolist() == [-1, -1]


def pin_slot_mapping_inverse(orc):
    w = small_decode(seed=11, ctx=(3, 17, 40))
    rows = np.concatenate([np.full(int(L), r) for r, L in enumerate(w.seq_lens)]).astype(np.int32)
    pos = np.concatenate([np.arange(int(L)) for L in w.seq_lens]).astype(np.int32)
    slots, bad = orc.slot_mapping(w.block_tables, w.num_blocks, rows, pos, w.block_size)
    assert bad == 0
    assert np.array_equal(slots // w.block_size, w.block_tables[rows, pos // w.block_size])
    assert np.array_equal(slots % w.block_size, pos % w.block_size)
    assert len(set(slots.tolist())) == len(slots) - _shared_positions(w)


def _shared_positions(w):
    # positions of the shared prefix are counted once per row but live once
    return w.shared_prefix_tokens * (w.batch - 1) if w.shared_prefix_tokens else 0


def pin_append_bit_exact(orc):
    for dtype in ("f32", "bf16"):
        w = small_decode(seed=13, dtype=dtype, ctx=(4, 9, 31), hkv=3, hq=6, d=8)
        kp, vp = appended(orc, w)
        ek, ev = w.k_pool.copy(), w.v_pool.copy()
        bs = w.block_size
        blk = w.block_tables[w.new_rows, w.new_pos // bs]
        ek[blk, :, w.new_pos % bs, :] = w.k_new
        ev[blk, :, w.new_pos % bs, :] = w.v_new
        assert kp.tobytes() == ek.tobytes() and vp.tobytes() == ev.tobytes()
    # negative slots are skipped and touch nothing
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    orc.append(kp, vp, w.dtype, np.full(w.new_rows.shape, -1, np.int32), w.k_new, w.v_new)
    assert kp.tobytes() == w.k_pool.tobytes() and vp.tobytes() == w.v_pool.tobytes()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def _decode_vs_dense(orc, w, rtol=1e-12):
    kp, vp = appended(orc, w)
    out = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window, w.scale)
    K, V, q = f64(kp, w.dtype), f64(vp, w.dtype), f64(w.q, w.dtype)
    G = w.num_q_heads // w.num_kv_heads
    for r in range(w.batch):
        L = int(w.seq_lens[r])
        lo = max(0, L - w.window) if w.window > 0 else 0
        for h in range(w.num_q_heads):
            g = h // G
            ref = dense_attention(q[r, h], gather_row(K, w.block_tables, r, g, lo, L, w.block_size),
                                  gather_row(V, w.block_tables, r, g, lo, L, w.block_size), w.scale)
            assert np.allclose(out[r, h], ref, rtol=rtol, atol=rtol), (r, h)


def pin_decode_paged_equals_flat(orc):
    _decode_vs_dense(orc, small_decode(seed=17, dtype="f32", hq=4, hkv=2, ctx=(1, 6, 23, 40)))
    _decode_vs_dense(orc, small_decode(seed=19, dtype="bf16", hq=8, hkv=2, ctx=(12, 31, 32, 47),
                                       prefix=12))
    _decode_vs_dense(orc, small_decode(seed=23, dtype="bf16", hq=3, hkv=3, ctx=(9, 50),
                                       window=7))
    _decode_vs_dense(orc, small_decode(seed=29, dtype="f32", hq=4, hkv=1, ctx=(30, 61),
                                       window=10, live_only=True))


def pin_decode_brute_force_mpmath(orc):
    import pytest
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    w = small_decode(seed=31, dtype="f32", hq=2, hkv=1, d=5, ctx=(6, 13), bs=4)
    kp, vp = appended(orc, w)
    out = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    for r in range(w.batch):
        L = int(w.seq_lens[r])
        for h in range(w.num_q_heads):
            qv = [mp.mpf(float(x)) for x in w.q[r, h]]
            s, vals = [], []
            for p in range(L):
                b = int(w.block_tables[r, p // 4])
                k = [mp.mpf(float(x)) for x in kp[b, 0, p % 4]]
                vals.append([mp.mpf(float(x)) for x in vp[b, 0, p % 4]])
                s.append(mp.mpf(w.scale) * mp.fsum(a * c for a, c in zip(qv, k)))
            e = [mp.exp(x) for x in s]
            z = mp.fsum(e)
            for d in range(w.head_dim):
                exact = mp.fsum(e[j] * vals[j][d] for j in range(L)) / z
                assert abs(float(exact) - out[r, h, d]) <= 1e-13 * (1 + abs(float(exact)))


def pin_decode_closed_forms(orc):
    bs = 4
    # one key: the output is that value exactly
    w = small_decode(seed=37, dtype="bf16", ctx=(0, 0), bs=bs)
    kp, vp = appended(orc, w)
    out = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    G = w.num_q_heads // w.num_kv_heads
    for r in range(w.batch):
        for h in range(w.num_q_heads):
            assert np.array_equal(out[r, h], f64(w.v_new[r, h // G], w.dtype))
    # zero query: the mean of the values in range (full and windowed)
    for window in (0, 5):
        w = small_decode(seed=41, dtype="f32", ctx=(9, 22), bs=bs, window=window)
        w.q[:] = 0
        kp, vp = appended(orc, w)
        out = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, window, w.scale)
        V = f64(vp, w.dtype)
        for r in range(w.batch):
            L = int(w.seq_lens[r])
            lo = max(0, L - window) if window else 0
            for h in range(w.num_q_heads):
                mean = gather_row(V, w.block_tables, r, h // G, lo, L, bs).mean(axis=0)
                assert np.allclose(out[r, h], mean, rtol=1e-13, atol=1e-13)
    # all keys equal: the mean of the values
    w = small_decode(seed=43, dtype="f32", ctx=(14,), bs=bs)
    w.k_pool[:] = w.k_pool[w.block_tables[0, 0], :, 0:1, :]
    w.k_new[:] = w.k_pool[w.block_tables[0, 0], :, 0, :]
    kp, vp = appended(orc, w)
    out = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    V = f64(vp, w.dtype)
    for h in range(w.num_q_heads):
        mean = gather_row(V, w.block_tables, 0, h // G, 0, 15, bs).mean(axis=0)
        assert np.allclose(out[0, h], mean, rtol=1e-13, atol=1e-13)
    # window 1: the newest value exactly; window >= length: full attention, bit for bit
    w = small_decode(seed=47, dtype="bf16", ctx=(3, 19), bs=bs)
    kp, vp = appended(orc, w)
    o1 = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 1, w.scale)
    for r in range(w.batch):
        for h in range(w.num_q_heads):
            assert np.array_equal(o1[r, h], f64(w.v_new[r, h // G], w.dtype))
    ofull = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    owide = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 20, w.scale)
    assert np.array_equal(ofull, owide)
    onarrow = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 19, w.scale)
    assert not np.array_equal(ofull[1], onarrow[1])  # 20 tokens, window 19 drops one
    # one dominant key (k = c q): its value
    w = small_decode(seed=53, dtype="f32", hq=1, hkv=1, d=16, ctx=(21,), bs=bs)
    j = 6
    b = w.block_tables[0, j // bs]
    w.k_pool[b, 0, j % bs, :] = 40.0 * w.q[0, 0]
    kp, vp = appended(orc, w)
    out = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    assert np.allclose(out[0, 0], vp[b, 0, j % bs], atol=1e-9)


def pin_decode_shared_equals_private(orc):
    w = small_decode(seed=59, dtype="bf16", hq=4, hkv=2, ctx=(8, 16, 29), prefix=8, bs=4)
    kp, vp = appended(orc, w)
    base = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 0, w.scale)
    P = w.shared_prefix_tokens // w.block_size
    nb = w.num_blocks
    extra = P * (w.batch - 1)
    kp2 = np.concatenate([kp, np.zeros((extra,) + kp.shape[1:], kp.dtype)])
    vp2 = np.concatenate([vp, np.zeros((extra,) + vp.shape[1:], vp.dtype)])
    t2 = w.block_tables.copy()
    k = nb
    for r in range(1, w.batch):
        for j in range(P):
            kp2[k], vp2[k] = kp[t2[r, j]], vp[t2[r, j]]
            t2[r, j] = k
            k += 1
    priv = orc.decode(w.q, kp2, vp2, w.dtype, t2, w.seq_lens, 0, w.scale)
    assert np.array_equal(base, priv)


def pin_decode_permutation_invariant(orc):
    w = small_decode(seed=61, dtype="bf16", hq=6, hkv=2, ctx=(5, 26, 43), bs=4)
    kp, vp = appended(orc, w)
    base = orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, 3, w.scale)
    perm = gen.permutation(99, "relabel", w.num_blocks)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out = orc.decode(w.q, kp2, vp2, w.dtype, t2, w.seq_lens, 3, w.scale)
    assert np.array_equal(base, out)


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def small_prefill(seed=67, dtype="bf16", hq=4, hkv=2, d=16, prefix=(0, 9, 20), chunk=(5, 1, 12),
                  window=0, bs=4):
    return gen.prefill_workload(seed=seed, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv,
                                head_dim=d, prefix_lens=list(prefix), chunk_lens=list(chunk),
                                block_size=bs, window=window)


def pin_prefill_equals_dense_causal(orc):
    for window in (0, 6):
        w = small_prefill(window=window)
        kp, vp = appended(orc, w)
        out = orc.prefill(w.q, w.cu_q_lens, kp, vp, w.dtype, w.block_tables, w.seq_lens, window,
                          w.scale)
        K, V, q = f64(kp, w.dtype), f64(vp, w.dtype), f64(w.q, w.dtype)
        G = w.num_q_heads // w.num_kv_heads
        for r in range(w.batch):
            c0, c1 = int(w.cu_q_lens[r]), int(w.cu_q_lens[r + 1])
            L = int(w.seq_lens[r])
            for i in range(c1 - c0):
                p = L - (c1 - c0) + i
                lo = max(0, p - window + 1) if window else 0
                for h in range(w.num_q_heads):
                    ref = dense_attention(q[c0 + i, h],
                                          gather_row(K, w.block_tables, r, h // G, lo, p + 1, w.block_size),
                                          gather_row(V, w.block_tables, r, h // G, lo, p + 1, w.block_size),
                                          w.scale)
                    assert np.allclose(out[c0 + i, h], ref, rtol=1e-12, atol=1e-12), (r, i, h)


def pin_prefill_row_equals_decode(orc):
    w = small_prefill(seed=71, prefix=(7, 16), chunk=(6, 3), window=5)
    kp, vp = appended(orc, w)
    out = orc.prefill(w.q, w.cu_q_lens, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window,
                      w.scale)
    for r in range(w.batch):
        c0, c1 = int(w.cu_q_lens[r]), int(w.cu_q_lens[r + 1])
        for i in range(c1 - c0):
            sl = w.seq_lens.copy()
            sl[r] = w.seq_lens[r] - (c1 - c0) + i + 1
            qd = np.repeat(w.q[c0 + i][None], w.batch, axis=0)
            dec = orc.decode(qd, kp, vp, w.dtype, w.block_tables, sl, w.window, w.scale,
                             pairs=np.array([[r, h] for h in range(w.num_q_heads)]))
            assert np.array_equal(out[c0 + i], dec)
    # the sampled form agrees with the full form
    s = np.array([[1, 2, 3], [0, 5, 0], [1, 0, 1]])
    samp = orc.prefill(w.q, w.cu_q_lens, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window,
                       w.scale, samples=s)
    for k, (r, i, h) in enumerate(s):
        assert np.array_equal(samp[k], out[w.cu_q_lens[r] + i, h])


# ---------------------------------------------------------------------------
# shared-prefix groups
# ---------------------------------------------------------------------------

def pin_prefix_groups_pages_example(orc):
    # "paged-cache.md", GDN ladder section: a 1400-token prompt at block size
    # 16 has its deepest full-block boundary at 1392 tokens = 87 blocks.
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "full_blocks_1400.txt")
    vals = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = int(v)
    bs, L, full = vals["block_size"], vals["prompt_tokens"], vals["full_block_tokens"]
    nblk = (L + bs - 1) // bs
    tables = np.tile(np.arange(nblk, dtype=np.int32), (2, 1))
    gor, pb = orc.prefix_groups(tables, np.array([L, L], np.int32), bs)
    assert gor.tolist() == [0, 0] and pb.tolist() == [full // bs]


def pin_prefix_groups_properties(orc):
    bs = 16
    t = np.array([[4, 7, 9, 1, -1],      # shares 2 blocks with rows 2, 4
                  [3, 8, -1, -1, -1],    # alone
                  [4, 7, 5, -1, -1],
                  [6, 2, 0, 10, 11],     # shares 3 blocks with row 5, but row 5 has 2 full
                  [4, 7, 9, 12, -1],
                  [6, 2, 0, 13, -1]], dtype=np.int32)
    L = np.array([60, 20, 40, 80, 64, 47], dtype=np.int32)
    gor, pb = orc.prefix_groups(t, L, bs)
    assert gor.tolist() == [0, -1, 0, 1, 0, 1] and pb.tolist() == [2, 2]
    # random tables: defining properties
    for seed in range(5):
        u = gen.uniform_ints(500 + seed, "t", 24 * 6, 0, 5).reshape(24, 6).astype(np.int32)
        Ls = gen.uniform_ints(600 + seed, "l", 24, 1, 96).astype(np.int32)
        gor, pb = orc.prefix_groups(u, Ls, bs)
        for gid in range(len(pb)):
            rows = np.nonzero(gor == gid)[0]
            P = int(pb[gid])
            assert len(rows) >= 2 and P >= 1
            assert all(np.array_equal(u[r, :P], u[rows[0], :P]) for r in rows)
            assert all(P * bs <= Ls[r] for r in rows)
            can_grow = P < u.shape[1] and all(u[r, P] == u[rows[0], P] for r in rows) \
                and all((P + 1) * bs <= Ls[r] for r in rows)
            assert not can_grow
        for r in np.nonzero(gor < 0)[0]:
            same = [s for s in range(24) if s != r and u[s, 0] == u[r, 0]]
            # alone, or sharing the first block only with rows grouped elsewhere
            # is impossible: rows with equal first blocks are grouped together
            assert not same or all(gor[s] < 0 for s in same)


# ---------------------------------------------------------------------------
# FP8 (E4M3) pools
# ---------------------------------------------------------------------------

def pin_e4m3_published_values(orc):
    # the E4M3 column of the format table in "FP8 Formats for Deep Learning"
    # (Micikevicius et al. 2022): bias 7, max normal S.1111.110 = 448, min
    # normal S.0001.000 = 2^-6, max subnormal S.0000.111 = 0.875 * 2^-6, min
    # subnormal S.0000.001 = 2^-9, NaN S.1111.111, no infinities
    codes = np.array([0x7E, 0x08, 0x07, 0x01, 0x38, 0xC0, 0x00], np.uint8)
    want = [448.0, 2.0 ** -6, 0.875 * 2.0 ** -6, 2.0 ** -9, 1.0, -2.0, 0.0]
    assert orc.e4m3_decode(codes).tolist() == want
    assert np.isnan(orc.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    negz = orc.e4m3_decode(np.array([0x80], np.uint8))[0]
    assert negz == 0.0 and math.copysign(1.0, negz) < 0


def pin_e4m3_grid_and_round_trip(orc):
    v = orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    # 3 mantissa bits: steps of 2^-9 through the subnormals and the first
    # binade, then the step doubles with every binade
    steps = np.diff(v)
    for c in range(0x7E):
        e = max(c >> 3, 1)   # binade of the lower code
        assert steps[c] == 2.0 ** (e - 10), c
    neg = orc.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -v)
    # every finite code is its own nearest code
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    x = orc.e4m3_decode(codes).astype(np.float32)
    x[codes == 0x80] = np.float32(-0.0)
    assert np.array_equal(orc.e4m3_encode(x), codes)


def pin_e4m3_rounding(orc):
    # worked cases: ties go to the even code, magnitudes past 448 saturate
    x = np.array([1.0625, 1.1875, 2.0 ** -10, -(2.0 ** -10), 3 * 2.0 ** -11, 460.0, 1e6, -1e6,
                  np.inf, 1.0 / 3.0, 0.0], np.float32)
    want = [0x38, 0x3A, 0x00, 0x80, 0x01, 0x7E, 0x7E, 0xFE, 0x7E, 0x2B, 0x00]
    assert orc.e4m3_encode(x).tolist() == want
    # every midpoint between neighbouring codes goes to the even one
    v = orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mid = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (v[:-1] + v[1:]) / 2)   # exact in float32
    got = orc.e4m3_encode(mid).astype(int)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))
    # off the midpoints the code is the nearest value (brute force over the grid)
    r = gen.uniform(gen.stream_seed(5, "e4m3"), 4000)
    x = (np.where(r[:2000] < 0.5, -1.0, 1.0) * 2.0 ** (r[2000:] * 22 - 12)).astype(np.float32)
    c = orc.e4m3_encode(x)
    dist = np.abs(np.abs(x.astype(np.float64))[:, None] - v[None, :])
    assert np.array_equal(c & 0x7F, np.argmin(dist, axis=1).astype(np.uint8))
    assert np.array_equal(c >> 7, (x < 0).astype(np.uint8))


def _mma_b_fragment(lane: int, i: int):
    """Row k and column n of element i (0..3) of the B fragment that thread
    `lane` holds in mma.m16n8k16 with 16-bit operands (PTX ISA, the figure of
    the B fragment layout for .f16/.bf16): groupID = lane / 4,
    threadID_in_group = lane % 4, k = threadID_in_group * 2 + (i % 2) + 8 * (i >= 2),
    n = groupID."""
    return (lane % 4) * 2 + (i % 2) + (8 if i >= 2 else 0), lane // 4


def fp8_tile_map(D: int):
    """(token, dim) of every byte of an FP8 K tile and V tile, from the
    fragment table: the K tile is the B operand of Q K^T (k = dim, n = token;
    per 64 dims two halves of 8 tokens, each lane's 16 bytes = its fragments
    of the four 16-dim steps), the V tile that of P V (k = token, n = dim;
    per 32 dims each lane's 16 bytes = its fragments of the four 8-dim steps)."""
    kt, kd, vt, vd = (np.full(16 * D, -1) for _ in range(4))
    for lane in range(32):
        for s in range(4):
            for i in range(4):
                k, n = _mma_b_fragment(lane, i)
                for grp in range(D // 64):
                    for half in range(2):
                        o = grp * 1024 + half * 512 + lane * 16 + s * 4 + i
                        kt[o], kd[o] = half * 8 + n, grp * 64 + s * 16 + k
                for grp in range(D // 32):
                    o = grp * 512 + lane * 16 + s * 4 + i
                    vt[o], vd[o] = k, grp * 32 + s * 8 + n
    return kt, kd, vt, vd


def fp8_dequantized(orc, pool: np.ndarray, scale, D: int, is_v: bool) -> np.ndarray:
    """An FP8 pool's values as float64 [nb, Hkv, 16, D] (code value * scale)."""
    kt, kd, vt, vd = fp8_tile_map(D)
    t, d = (vt, vd) if is_v else (kt, kd)
    vals = orc.e4m3_decode(pool) * float(scale)
    out = np.empty(pool.shape[:2] + (16, D))
    out[:, :, t, d] = vals
    return out


def pin_fp8_tile_layout(orc):
    # one token at a time into a fresh pool: the code of value 0x20 + d marks
    # where (t, d) lands
    for D in (64, 128):
        kt, kd, vt, vd = fp8_tile_map(D)
        assert sorted(zip(kt, kd)) == [(t, d) for t in range(16) for d in range(D)]
        assert sorted(zip(vt, vd)) == [(t, d) for t in range(16) for d in range(D)]
        codes = (0x20 + np.arange(D) % 64).astype(np.uint8)
        row = gen.bf16_bits(orc.e4m3_decode(codes).astype(np.float32)).reshape(1, 1, D)
        for t in range(16):
            kp = np.full((1, 1, 16 * D), 0x7F, np.uint8)
            vp = kp.copy()
            orc.append(kp, vp, "fp8", np.array([t], np.int32), row, row, 1.0, 1.0)
            for pool, (tt, dd) in ((kp, (kt, kd)), (vp, (vt, vd))):
                mine = tt == t
                assert np.array_equal(pool[0, 0, mine], codes[dd[mine]]), (D, t)
                assert (pool[0, 0, ~mine] == 0x7F).all()


def pin_fp8_append_quantizes(orc):
    w = small_decode(seed=37, dtype="bf16", hq=4, hkv=2, d=64, ctx=(5, 30), bs=16)
    kp, vp = gen.fp8_empty_pools(w)
    slots = oracle_slots(orc, w)
    ks, vs = gen.FP8_K_SCALE, gen.FP8_V_SCALE
    orc.append(kp, vp, "fp8", slots, w.k_new, w.v_new, ks, vs)
    kt, kd, vt, vd = fp8_tile_map(64)
    for i, s in enumerate(slots):
        b, t = divmod(int(s), 16)
        for pool, new, sc, (tt, dd) in ((kp, w.k_new, ks, (kt, kd)), (vp, w.v_new, vs, (vt, vd))):
            mine = tt == t
            q = gen.bf16_to_f32(new[i]) / np.float32(sc)         # float32 quotient
            assert q.dtype == np.float32
            assert np.array_equal(pool[b][:, mine], orc.e4m3_encode(q)[:, dd[mine]])
    touched = np.zeros(kp.shape[0], bool)
    touched[slots // 16] = True
    assert (kp[~touched] == 0x7F).all() and (vp[~touched] == 0x7F).all()


def _fp8_context(orc, w):
    kp, vp = gen.fp8_empty_pools(w)
    ks, vs = gen.FP8_K_SCALE, gen.FP8_V_SCALE
    s, kr, vr = gen.live_slots(w)
    orc.append(kp, vp, "fp8", s, kr, vr, ks, vs)
    orc.append(kp, vp, "fp8", oracle_slots(orc, w), w.k_new, w.v_new, ks, vs)
    return kp, vp


def pin_fp8_decode_equals_dense(orc):
    for seed, ctx, window, prefix in ((41, (1, 17, 40, 77), 0, 0), (43, (33, 64, 90), 20, 32)):
        w = small_decode(seed=seed, dtype="bf16", hq=8, hkv=2, d=64, ctx=ctx, bs=16,
                         window=window, prefix=prefix)
        kp, vp = _fp8_context(orc, w)
        out = orc.decode(w.q, kp, vp, "fp8", w.block_tables, w.seq_lens, w.window, w.scale,
                         k_scale=gen.FP8_K_SCALE, v_scale=gen.FP8_V_SCALE)
        K = fp8_dequantized(orc, kp, gen.FP8_K_SCALE, 64, False)
        V = fp8_dequantized(orc, vp, gen.FP8_V_SCALE, 64, True)
        q = f64(w.q, "bf16")
        for r in range(w.batch):
            L = int(w.seq_lens[r])
            lo = max(0, L - w.window) if w.window > 0 else 0
            for h in range(w.num_q_heads):
                g = h // 4
                ref = dense_attention(q[r, h], gather_row(K, w.block_tables, r, g, lo, L, 16),
                                      gather_row(V, w.block_tables, r, g, lo, L, 16), w.scale)
                assert np.allclose(out[r, h], ref, rtol=1e-12, atol=1e-12), (seed, r, h)


def pin_fp8_prefill_equals_dense_causal(orc):
    w = gen.prefill_workload(seed=47, dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=64,
                             prefix_lens=[0, 21, 40], chunk_lens=[9, 16, 3])
    kp, vp = _fp8_context(orc, w)
    out = orc.prefill(w.q, w.cu_q_lens, kp, vp, "fp8", w.block_tables, w.seq_lens, 0, w.scale,
                      k_scale=gen.FP8_K_SCALE, v_scale=gen.FP8_V_SCALE)
    K = fp8_dequantized(orc, kp, gen.FP8_K_SCALE, 64, False)
    V = fp8_dequantized(orc, vp, gen.FP8_V_SCALE, 64, True)
    q = f64(w.q, "bf16")
    for r in range(w.batch):
        c0, c1, L = int(w.cu_q_lens[r]), int(w.cu_q_lens[r + 1]), int(w.seq_lens[r])
        for i in range(c1 - c0):
            p = L - (c1 - c0) + i
            for h in range(4):
                ref = dense_attention(q[c0 + i, h], gather_row(K, w.block_tables, r, h // 2, 0, p + 1, 16),
                                      gather_row(V, w.block_tables, r, h // 2, 0, p + 1, 16), w.scale)
                assert np.allclose(out[c0 + i, h], ref, rtol=1e-12, atol=1e-12), (r, i, h)


ALL_PINS = [
    pin_slot_mapping_hand_worked,
    pin_slot_mapping_inverse,
    pin_append_bit_exact,
    pin_decode_paged_equals_flat,
    pin_decode_brute_force_mpmath,
    pin_decode_closed_forms,
    pin_decode_shared_equals_private,
    pin_decode_permutation_invariant,
    pin_prefill_equals_dense_causal,
    pin_prefill_row_equals_decode,
    pin_prefix_groups_pages_example,
    pin_prefix_groups_properties,
    pin_e4m3_published_values,
    pin_e4m3_grid_and_round_trip,
    pin_e4m3_rounding,
    pin_fp8_tile_layout,
    pin_fp8_append_quantizes,
    pin_fp8_decode_equals_dense,
    pin_fp8_prefill_equals_dense_causal,
]
