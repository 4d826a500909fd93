"""Helpers for the GPU parity tests: upload a workload, run the library's
append + decode / prefill through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import pkv_inputs as gen

BF16_ATOL, BF16_RTOL = 2e-3, 1e-2   # bf16 K/V, fp32 accumulation
F32_ATOL, F32_RTOL = 1e-5, 1e-5


def tol(dtype: str):
    return (BF16_ATOL, BF16_RTOL) if dtype == "bf16" else (F32_ATOL, F32_RTOL)


def to_torch(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def storage_bytes(t: torch.Tensor) -> bytes:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes()


class Dev:
    """A workload's arrays on the GPU."""

    def __init__(self, w: gen.Workload, device="cuda"):
        self.w = w
        self.k_pool = to_torch(w.k_pool, w.dtype, device)
        self.v_pool = to_torch(w.v_pool, w.dtype, device)
        self.q = to_torch(w.q, w.dtype, device)
        self.k_new = to_torch(w.k_new, w.dtype, device)
        self.v_new = to_torch(w.v_new, w.dtype, device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(device)
        self.cu = torch.from_numpy(w.cu_q_lens).to(device) if w.cu_q_lens is not None else None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)


def append(pkv, d: Dev) -> np.ndarray:
    w = d.w
    slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                  w.block_size)
    pkv.paged_kv_append(d.k_pool, d.v_pool, torch.from_numpy(slots).to(d.k_pool.device),
                        d.k_new, d.v_new, status=d.status)
    return slots


def oracle_pools(orc, w: gen.Workload):
    slots, bad = orc.slot_mapping(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                  w.block_size)
    assert bad == 0
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    orc.append(kp, vp, w.dtype, slots, w.k_new, w.v_new)
    return slots, kp, vp


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    atol, rtol = tol(dtype)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside |d| <= {atol} + {rtol}|ref| "
            f"(max abs {err.max():.3g}); first {idx.tolist()} got {got[bad][:5]} ref {ref[bad][:5]}")


def sample_pairs(w: gen.Workload, n: int, seed: int = 0) -> np.ndarray:
    """(row, head) pairs: every row's first and last head plus seeded extras."""
    pairs = {(r, 0) for r in range(w.batch)} | {(r, w.num_q_heads - 1) for r in range(w.batch)}
    u = gen.uniform_ints(seed, "pairs", 2 * n, 0, 1 << 30)
    for i in range(n):
        pairs.add((int(u[2 * i]) % w.batch, int(u[2 * i + 1]) % w.num_q_heads))
    return np.array(sorted(pairs), dtype=np.int32)


def assert_appended_blocks_equal(d: Dev, slots: np.ndarray, kp: np.ndarray, vp: np.ndarray):
    """Every pool block that received a token of the append, K and V, equals
    the oracle's byte for byte (the new rows and the untouched rows beside
    them): the pool check of workloads too large to copy back whole."""
    bs = d.w.block_size
    blocks = np.unique(slots[slots >= 0] // bs)
    idx = torch.from_numpy(blocks.astype(np.int64)).to(d.k_pool.device)
    for got, ref, name in ((d.k_pool, kp, "K"), (d.v_pool, vp, "V")):
        g = got.index_select(0, idx).contiguous().view(torch.uint8).cpu().numpy().tobytes()
        r = np.ascontiguousarray(ref[blocks]).tobytes()
        assert g == r, f"{name} pool blocks of the appended tokens differ from the oracle's"


def oracle_decode_rows(orc, q, kp, vp, dtype, tables, seq_lens, window, scale, num_q_heads,
                       threads=None, **kw):
    """The oracle's full [B, Hq, D] decode output, one row per oracle call on
    a pool of host threads (the oracle's C calls release the interpreter
    lock); the same arithmetic as one call over the whole batch."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    batch = tables.shape[0]

    def one(r):
        pairs = np.array([[r, h] for h in range(num_q_heads)], dtype=np.int32)
        return orc.decode(q, kp, vp, dtype, tables, seq_lens, window, scale, pairs=pairs, **kw)

    with ThreadPoolExecutor(max_workers=threads or os.cpu_count() or 1) as ex:
        rows = list(ex.map(one, range(batch)))
    return np.stack(rows)
