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
