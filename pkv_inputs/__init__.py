"""Seeded synthetic inputs for the paged-KV attention path.

This module only draws numbers and lays out which physical pool block holds
which logical block of each request. It holds none of the attention, append,
slot-mapping or prefix-grouping arithmetic: those live, written twice and
independently, in the CUDA library and in the CPU oracle, and both receive
exactly the arrays built here.

Generator (stated so that any other implementation can reproduce it):
  * SplitMix64, counter based: for stream seed ``s`` and counter ``i`` the
    64-bit word is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)`` with the usual
    SplitMix64 finaliser (xor-shift 30/27/31, multipliers 0xBF58476D1CE4E5B9
    and 0x94D049BB133111EB), all mod 2**64.
  * uniform in [0, 1): ``(word >> 11) * 2**-53``.
  * N(0, 1): Box-Muller on consecutive pairs ``(u1, u2)``:
    ``r = sqrt(-2 ln(1 - u1))``, values ``r cos(2 pi u2)`` and ``r sin(2 pi u2)``,
    computed in float64 and rounded to float32.
  * bf16: round-to-nearest-even of the float32 bit pattern (top 16 bits).
  * permutation: Fisher-Yates, ``j = floor(u * (i + 1))`` for i = n-1 .. 1.
  * each named array draws from its own stream ``s = mix(seed) ^ fnv1a64(name)``.

Workload recipes follow the pages' setting: block size 16 (the value used
throughout "paged-cache.md"), K/V pools laid out ``[block][kv_head][slot][dim]``,
refcounted shared prefix blocks (one physical block referenced by several block
tables), sliding groups whose expired logical blocks hold the null sentinel -1
("paged-cache.md", Gemma4 coordinator section), and a query chunk whose K/V is
appended before attention (chunked prefill, "paged-cache.md" GDN ladder section
and the MLX_PAGED_PREFILL_CHUNK_SIZE knob of "perf.md").
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB

BF16_NAN = 0x7FC0
F32_NAN = np.float32("nan")


def _mix_scalar(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * _C1) & M64
    z = ((z ^ (z >> 27)) * _C2) & M64
    return z ^ (z >> 31)


def _fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for b in name.encode():
        h = ((h ^ b) * 0x100000001B3) & M64
    return h


def stream_seed(seed: int, name: str) -> int:
    """Seed of the named stream derived from a workload seed."""
    return _mix_scalar(seed) ^ _fnv1a64(name)


def splitmix64(s: int, start: int, n: int) -> np.ndarray:
    """Words ``start .. start+n-1`` of the counter-based SplitMix64 stream ``s``."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(s & M64) + i * np.uint64(_GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_C1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_C2)
        z = z ^ (z >> np.uint64(31))
    return z


def uniform(s: int, n: int, start: int = 0) -> np.ndarray:
    return (splitmix64(s, start, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_CHUNK = 1 << 22


def normal_f32(seed: int, name: str, n: int) -> np.ndarray:
    """``n`` float32 N(0,1) values of the named stream (Box-Muller, see module doc)."""
    s = stream_seed(seed, name)
    npairs = (n + 1) // 2
    out = np.empty(2 * npairs, dtype=np.float32)
    for p0 in range(0, npairs, _CHUNK):
        m = min(_CHUNK, npairs - p0)
        u = uniform(s, 2 * m, start=2 * p0)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * math.pi * u2
        out[2 * p0:2 * (p0 + m):2] = (r * np.cos(t)).astype(np.float32)
        out[2 * p0 + 1:2 * (p0 + m):2] = (r * np.sin(t)).astype(np.float32)
    return out[:n]


def uniform_ints(seed: int, name: str, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform on the closed range [lo, hi]."""
    u = uniform(stream_seed(seed, name), n)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def permutation(seed: int, name: str, n: int) -> np.ndarray:
    """Fisher-Yates permutation of 0..n-1 driven by the named stream."""
    p = np.arange(n, dtype=np.int64)
    if n < 2:
        return p
    u = uniform(stream_seed(seed, name), n - 1)
    for k, i in enumerate(range(n - 1, 0, -1)):
        j = int(u[k] * (i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the exact float32 values."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _values(seed: int, name: str, shape, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    v = normal_f32(seed, name, n).reshape(shape)
    return bf16_bits(v) if dtype == "bf16" else v


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array (float32 or bf16 bits) -> float32 values."""
    return bf16_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


@dataclasses.dataclass
class Workload:
    """One paged attention call with its append.

    Arrays are host numpy arrays in storage form: float32, or uint16 bf16 bits.
    ``seq_lens`` counts every token of a row including those appended by this
    step; the appended tokens sit at absolute positions ``new_pos`` of rows
    ``new_rows`` and their pool slots are poisoned (NaN) until the append.
    """
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    window: int
    scale: float
    k_pool: np.ndarray          # [num_blocks, Hkv, bs, D]
    v_pool: np.ndarray
    q: np.ndarray               # decode: [B, Hq, D]; prefill: [sum C, Hq, D]
    block_tables: np.ndarray    # int32 [B, max_blocks_per_seq], -1 = none / null sentinel
    seq_lens: np.ndarray        # int32 [B]
    new_rows: np.ndarray        # int32 [T]
    new_pos: np.ndarray         # int32 [T]
    k_new: np.ndarray           # [T, Hkv, D]
    v_new: np.ndarray
    cu_q_lens: Optional[np.ndarray] = None   # prefill only: int32 [B+1]
    shared_prefix_tokens: int = 0            # as built (the library derives its own descriptor)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


def _build(*, name: str, seed: int, dtype: str, num_q_heads: int, num_kv_heads: int,
           head_dim: int, block_size: int, context_lens: Sequence[int],
           new_per_row: Sequence[int], shared_prefix_tokens: int = 0, window: int = 0,
           pool_blocks: Optional[int] = None, table_width: Optional[int] = None,
           sliding_live_only: bool = False, poison: bool = True,
           prefill: bool = False) -> Workload:
    assert dtype in ("f32", "bf16")
    assert num_q_heads % num_kv_heads == 0
    bs = block_size
    B = len(context_lens)
    ctx = np.asarray(context_lens, dtype=np.int64)
    nnew = np.asarray(new_per_row, dtype=np.int64)
    L = ctx + nnew
    assert shared_prefix_tokens % bs == 0, "a shared prefix is whole blocks"
    P = shared_prefix_tokens // bs
    assert np.all(ctx >= shared_prefix_tokens), "rows hold at least the shared prefix"
    nblk = (L + bs - 1) // bs
    width = int(table_width if table_width is not None else max(1, int(nblk.max(initial=0))))
    assert width >= int(nblk.max(initial=0))

    # logical blocks that hold data: with sliding_live_only, blocks wholly
    # before the window hold the null sentinel and own no pool block.
    first_live = np.zeros(B, dtype=np.int64)
    if sliding_live_only and window > 0:
        lo = np.maximum(0, L - window)
        first_live = lo // bs
        assert P == 0, "a sliding group here carries no shared prefix"
    private = [int(nblk[r] - max(P, first_live[r])) for r in range(B)]
    need = P + sum(private)
    nb = int(pool_blocks if pool_blocks is not None else need)
    assert nb >= need, (nb, need)
    perm = permutation(seed, "block_ids", nb)

    tables = np.full((B, width), -1, dtype=np.int32)
    k = 0
    for j in range(P):
        tables[:, j] = perm[k]
        k += 1
    for r in range(B):
        for j in range(max(P, int(first_live[r])), int(nblk[r])):
            tables[r, j] = perm[k]
            k += 1

    Hkv, D = num_kv_heads, head_dim
    shape = (nb, Hkv, bs, D)
    k_pool = _values(seed, "k_pool", shape, dtype)
    v_pool = _values(seed, "v_pool", shape, dtype)
    if poison:
        nan = BF16_NAN if dtype == "bf16" else F32_NAN
        used = np.zeros(nb, dtype=bool)
        used[tables[tables >= 0]] = True
        k_pool[~used] = nan
        v_pool[~used] = nan
        for r in range(B):
            # every slot at or past the existing context (the append targets
            # and the tail of the last block) holds stale data
            for p in range(int(ctx[r]), int(nblk[r] * bs)):
                b = tables[r, p // bs]
                k_pool[b, :, p % bs, :] = nan
                v_pool[b, :, p % bs, :] = nan

    rows = np.repeat(np.arange(B, dtype=np.int32), nnew)
    pos = np.concatenate([np.arange(ctx[r], L[r]) for r in range(B)]).astype(np.int32) \
        if int(nnew.sum()) else np.zeros(0, dtype=np.int32)
    T = int(nnew.sum())
    k_new = _values(seed, "k_new", (T, Hkv, D), dtype)
    v_new = _values(seed, "v_new", (T, Hkv, D), dtype)
    if prefill:
        q = _values(seed, "q", (T, num_q_heads, D), dtype)
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(nnew)
    else:
        q = _values(seed, "q", (B, num_q_heads, D), dtype)
        cu = None
    return Workload(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=Hkv,
                    head_dim=D, block_size=bs, num_blocks=nb, window=window,
                    scale=1.0 / math.sqrt(D), k_pool=k_pool, v_pool=v_pool, q=q,
                    block_tables=tables, seq_lens=L.astype(np.int32), new_rows=rows,
                    new_pos=pos, k_new=k_new, v_new=v_new, cu_q_lens=cu,
                    shared_prefix_tokens=shared_prefix_tokens)


def decode_workload(*, seed: int, dtype: str, num_q_heads: int, num_kv_heads: int,
                    head_dim: int, context_lens: Sequence[int], block_size: int = 16,
                    shared_prefix_tokens: int = 0, window: int = 0,
                    pool_blocks: Optional[int] = None, table_width: Optional[int] = None,
                    sliding_live_only: bool = False, poison: bool = True,
                    name: str = "decode") -> Workload:
    """Decode step: one new token per row appended at position ``context_lens[r]``."""
    return _build(name=name, seed=seed, dtype=dtype, num_q_heads=num_q_heads,
                  num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                  context_lens=context_lens, new_per_row=[1] * len(context_lens),
                  shared_prefix_tokens=shared_prefix_tokens, window=window,
                  pool_blocks=pool_blocks, table_width=table_width,
                  sliding_live_only=sliding_live_only, poison=poison)


def prefill_workload(*, seed: int, dtype: str, num_q_heads: int, num_kv_heads: int,
                     head_dim: int, prefix_lens: Sequence[int], chunk_lens: Sequence[int],
                     block_size: int = 16, window: int = 0, shared_prefix_tokens: int = 0,
                     pool_blocks: Optional[int] = None, poison: bool = True,
                     name: str = "prefill") -> Workload:
    """Chunked prefill: row r's chunk of ``chunk_lens[r]`` queries follows its
    ``prefix_lens[r]`` cached tokens; the chunk's K/V is appended first."""
    return _build(name=name, seed=seed, dtype=dtype, num_q_heads=num_q_heads,
                  num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                  context_lens=prefix_lens, new_per_row=chunk_lens,
                  shared_prefix_tokens=shared_prefix_tokens, window=window,
                  pool_blocks=pool_blocks, poison=poison, prefill=True)


# ---------------------------------------------------------------------------
# FP8 pools
# ---------------------------------------------------------------------------

# per-layer scales of the FP8 K and V pools ("perf.md" quantisation table: the
# paged adapter's FP8 KV cache keeps one scale per layer); deliberately not
# powers of two, so that the quotient's rounding matters
FP8_K_SCALE = np.float32(0.0123)
FP8_V_SCALE = np.float32(0.0171)
FP8_POISON = 0x7F   # the E4M3 NaN code: what an FP8 pool holds before any write


def live_slots(w: Workload):
    """Every pool slot that holds context in ``w`` (not poisoned, not one of
    this step's append targets) with its K and V rows: ``(slots, k_rows,
    v_rows)``, rows ``[n, Hkv, D]`` in storage form.  An FP8 pool is filled by
    appending exactly these rows, so that it holds the same context as the
    bf16 pool of the workload."""
    live = ~np.isnan(as_f32(w.k_pool[:, 0, :, 0], w.dtype))
    b, t = np.nonzero(live)
    slots = (b * w.block_size + t).astype(np.int32)
    return slots, np.ascontiguousarray(w.k_pool[b, :, t, :]), np.ascontiguousarray(w.v_pool[b, :, t, :])


def fp8_empty_pools(w: Workload):
    """Two FP8 pools for ``w`` (uint8 tile bytes ``[nb, Hkv, 16 * D]``), every
    byte the poison code."""
    assert w.block_size == 16
    shape = (w.num_blocks, w.num_kv_heads, 16 * w.head_dim)
    return np.full(shape, FP8_POISON, np.uint8), np.full(shape, FP8_POISON, np.uint8)


# ---------------------------------------------------------------------------
# The five workloads (seed = 1000 + index)
# ---------------------------------------------------------------------------

def tiny_f32() -> Workload:
    """fp32, 2 rows of 37 and 50 tokens (after the append) sharing a 2-block
    prefix, 4 q heads / 2 kv heads, head_dim 64, a 16-block pool."""
    return decode_workload(seed=1000, dtype="f32", num_q_heads=4, num_kv_heads=2,
                           head_dim=64, context_lens=[36, 49], shared_prefix_tokens=32,
                           pool_blocks=16, name="tiny_f32_b2_h4x2_d64")


def dense_bf16() -> Workload:
    """bf16, batch 4 x 2048 tokens, 16 q / 8 kv heads, head_dim 128, block
    tables drawn from a 2048-block pool."""
    return decode_workload(seed=1001, dtype="bf16", num_q_heads=16, num_kv_heads=8,
                           head_dim=128, context_lens=[2047] * 4, pool_blocks=2048,
                           name="dense_bf16_b4_ctx2048_h16x8_d128")


def shared_prefix_suffix_lens(seed: int = 1002, batch: int = 32, max_suffix: int = 7168) -> List[int]:
    return [int(x) for x in uniform_ints(seed, "suffix_lens", batch, 0, max_suffix)]


def shared_prefix_b32(batch: int = 32, max_suffix: int = 7168, prefix_tokens: int = 1024) -> Workload:
    """bf16, batch 32, 32 q / 8 kv heads, head_dim 128; a 1024-token prefix
    (64 blocks) shared by every row plus private suffixes uniform on 0..7168."""
    suf = shared_prefix_suffix_lens(1002, batch, max_suffix)
    return decode_workload(seed=1002, dtype="bf16", num_q_heads=32, num_kv_heads=8,
                           head_dim=128, context_lens=[prefix_tokens + s for s in suf],
                           shared_prefix_tokens=prefix_tokens,
                           name=f"shared_prefix_bf16_b{batch}_p{prefix_tokens}_s0-{max_suffix}_h32x8_d128")


def long_two_groups(batch: int = 4, context: int = 32768, window: int = 512):
    """bf16, batch 4 at 32768 tokens, 8 q / 1 kv head, head_dim 256: a full
    attention group and a sliding-window group (window 512) in separate pools."""
    full = decode_workload(seed=1003, dtype="bf16", num_q_heads=8, num_kv_heads=1,
                           head_dim=256, context_lens=[context - 1] * batch,
                           name=f"long_full_bf16_b{batch}_ctx{context}_h8x1_d256")
    nlive = window // 16 + 1
    sliding = decode_workload(seed=2003, dtype="bf16", num_q_heads=8, num_kv_heads=1,
                              head_dim=256, context_lens=[context - 1] * batch,
                              window=window, sliding_live_only=True,
                              pool_blocks=batch * nlive,
                              name=f"long_sliding_bf16_b{batch}_ctx{context}_w{window}_h8x1_d256")
    return full, sliding


def verify_steps(batch: int = 32, q_len: int = 4, min_ctx: int = 1024,
                 max_ctx: int = 8192) -> Workload:
    """bf16, 32 rows, each a speculative-verify step of 4 queries after a paged
    context uniform on 1024..8192 tokens, 32 q / 8 kv heads, head_dim 128."""
    ctx = [int(x) for x in uniform_ints(1005, "verify_ctx", batch, min_ctx, max_ctx)]
    return prefill_workload(seed=1005, dtype="bf16", num_q_heads=32, num_kv_heads=8,
                            head_dim=128, prefix_lens=ctx, chunk_lens=[q_len] * batch,
                            name=f"verify_bf16_b{batch}_q{q_len}_ctx{min_ctx}-{max_ctx}_h32x8_d128")


def chunked_prefill(batch: int = 4, chunk: int = 512, prefix: int = 16384) -> Workload:
    """bf16, 4 rows, a 512-query chunk each after a 16384-token paged prefix,
    32 q / 8 kv heads, head_dim 128, causal within the chunk."""
    return prefill_workload(seed=1004, dtype="bf16", num_q_heads=32, num_kv_heads=8,
                            head_dim=128, prefix_lens=[prefix] * batch,
                            chunk_lens=[chunk] * batch,
                            name=f"chunked_prefill_bf16_b{batch}_c{chunk}_p{prefix}_h32x8_d128")
