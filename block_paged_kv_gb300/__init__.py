"""GB300-native block-paged KV attention: Python binding of ``libpkv.so``.

The functions here only marshal arguments (torch tensors -> device pointers,
sizes and the current CUDA stream) into the C ABI declared in
``include/pkv.h``; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing, importing
this package raises.

Layouts (see ``include/pkv.h``): pools ``[num_blocks, num_kv_heads,
block_size, head_dim]``; ``q``/``out`` ``[batch, num_q_heads, head_dim]``
(prefill: ``[sum C, num_q_heads, head_dim]``); block tables int32
``[batch, max_blocks_per_seq]``; ``seq_lens`` int32 ``[batch]`` counting the
tokens appended this step.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_WORKSPACE, PKV_ERR_OUT_OF_BLOCKS = range(6)
PKV_F32, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_LEN, DEV_BAD_PREFIX, DEV_TIMEOUT = 1, 2, 4, 8, 16
DEV_Q_RANGE = 32

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it first "
                      "(python -c 'import __graft_entry__ as g; g.build()')")
_lib = ctypes.CDLL(LIB_PATH)


class _Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class _Prefix(ctypes.Structure):
    _fields_ = [("num_groups", ctypes.c_int32), ("max_group_rows", ctypes.c_int32),
                ("max_prefix_blocks", ctypes.c_int32), ("group_of_row", ctypes.c_void_p),
                ("prefix_blocks", ctypes.c_void_p)]


class _Group(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("out", ctypes.c_void_p), ("pool", _Pool),
                ("block_tables", ctypes.c_void_p), ("max_blocks_per_seq", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("max_seq_len", ctypes.c_int32),
                ("window", ctypes.c_int32), ("scale", ctypes.c_float)]


MAX_DECODE_GROUPS = 4

_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_PP, _XP = ctypes.POINTER(_Pool), ctypes.POINTER(_Prefix)
_GP = ctypes.POINTER(_Group)

_lib.paged_kv_append.argtypes = [_PP, _vp, _i32, _vp, _vp, _vp, _vp]
_lib.paged_kv_append.restype = ctypes.c_int
_lib.paged_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _XP]
_lib.paged_decode_workspace_size.restype = _sz
_lib.paged_decode_attention.argtypes = [_vp, _i32, _PP, _vp, _i32, _vp, _i32, _i32, _i32,
                                        ctypes.c_float, _vp, _vp, _sz, _XP, _vp, _vp]
_lib.paged_decode_attention.restype = ctypes.c_int
_lib.paged_decode_groups_workspace_size.argtypes = [_GP, _i32, _i32, _i32]
_lib.paged_decode_groups_workspace_size.restype = _sz
_lib.paged_decode_attention_groups.argtypes = [_GP, _i32, _i32, _i32, _vp, _sz, _vp, _vp]
_lib.paged_decode_attention_groups.restype = ctypes.c_int
_lib.paged_prefill_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]
_lib.paged_prefill_workspace_size.restype = _sz
_lib.paged_prefill_chunk_attention.argtypes = [_vp, _vp, _i32, _PP, _vp, _i32, _vp, _i32, _i32,
                                               _i32, _i32, ctypes.c_float, _vp, _vp, _sz, _vp, _vp]
_lib.paged_prefill_chunk_attention.restype = ctypes.c_int
_lib.pkv_status_string.argtypes = [ctypes.c_int]
_lib.pkv_status_string.restype = ctypes.c_char_p
_lib.pkv_slot_mapping_host.argtypes = [_vp, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp]
_lib.pkv_slot_mapping_host.restype = ctypes.c_int
_lib.pkv_prefix_groups_host.argtypes = [_vp, _i32, _vp, _i32, _i32, _vp, _vp]
_lib.pkv_prefix_groups_host.restype = _i32
_lib.pkv_set_decode_split_blocks.argtypes = [_i32]
_lib.pkv_set_decode_split_blocks.restype = _i32
_lib.pkv_set_wait_drill.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
_lib.pkv_set_wait_drill.restype = ctypes.c_int
_lib.pkv_decode_plan.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                 ctypes.POINTER(_i32)]
_lib.pkv_decode_plan.restype = _i32
_lib.pkv_version.restype = ctypes.c_char_p
_lib.pkv_profile_enable.argtypes = [ctypes.c_uint32]
_lib.pkv_profile_enable.restype = ctypes.c_int
_lib.pkv_profile_mask.argtypes = [ctypes.c_uint32]
_lib.pkv_profile_mask.restype = ctypes.c_int
_lib.pkv_profile_read.argtypes = [_i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)]
_lib.pkv_profile_read.restype = ctypes.c_int
_lib.pkv_profile_times.argtypes = [_i32, _vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]
_lib.pkv_profile_times.restype = ctypes.c_int
_lib.pkv_launch_count.restype = ctypes.c_int64
_lib.paged_decode_attention_no_alloc.argtypes = [_vp, _i32, _PP, _vp, _i32, _vp, _i32, _i32, _i32,
                                                 ctypes.c_float, _vp, _XP, _vp, _vp]
_lib.paged_decode_attention_no_alloc.restype = ctypes.c_int
NO_ALLOC_SCRATCH_BYTES = 16 << 20
_u64p = ctypes.POINTER(ctypes.c_uint64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_lib.pkv_slot_mapping_check_host.argtypes = [_vp, _i32, _i32, _i32, _i32p]
_lib.pkv_slot_mapping_check_host.restype = ctypes.c_int
_lib.pkv_allocator_create.argtypes = [_i32, _i32, _i32]
_lib.pkv_allocator_create.restype = _vp
_lib.pkv_allocator_destroy.argtypes = [_vp]
_lib.pkv_allocator_destroy.restype = None
_lib.pkv_allocator_begin.argtypes = [_vp]
_lib.pkv_allocator_begin.restype = _i32
_lib.pkv_allocator_find_cached_prefix.argtypes = [_vp, _i32, _vp, _i32, _vp, _i32p]
_lib.pkv_allocator_find_cached_prefix.restype = ctypes.c_int
_lib.pkv_allocator_reserve.argtypes = [_vp, _i32, _i32]
_lib.pkv_allocator_reserve.restype = ctypes.c_int
_lib.pkv_allocator_publish.argtypes = [_vp, _i32, _vp, _i32, _vp]
_lib.pkv_allocator_publish.restype = ctypes.c_int
_lib.pkv_allocator_expire.argtypes = [_vp, _i32, _i32]
_lib.pkv_allocator_expire.restype = ctypes.c_int
_lib.pkv_allocator_release.argtypes = [_vp, _i32]
_lib.pkv_allocator_release.restype = ctypes.c_int
_lib.pkv_allocator_table.argtypes = [_vp, _i32, _vp, _i32, _i32p]
_lib.pkv_allocator_table.restype = ctypes.c_int
_lib.pkv_allocator_refcount.argtypes = [_vp, _i32]
_lib.pkv_allocator_refcount.restype = _i32
_lib.pkv_allocator_stats.argtypes = [_vp, _i32p, _i32p, _i32p, _i32p]
_lib.pkv_allocator_stats.restype = ctypes.c_int

KERNEL_APPEND, KERNEL_DECODE_PREFIX, KERNEL_DECODE_SPLIT, KERNEL_DECODE_COMBINE, KERNEL_PREFILL = range(5)

EXPORTED = ["paged_kv_append", "paged_decode_workspace_size", "paged_decode_attention",
            "paged_prefill_workspace_size", "paged_prefill_chunk_attention", "pkv_status_string",
            "pkv_slot_mapping_host", "pkv_slot_mapping_check_host", "pkv_prefix_groups_host",
            "pkv_set_decode_split_blocks", "pkv_set_wait_drill",
            "pkv_decode_plan", "pkv_version", "pkv_profile_enable", "pkv_profile_mask", "pkv_profile_read", "pkv_profile_times",
            "pkv_launch_count", "paged_decode_attention_no_alloc", "paged_decode_groups_workspace_size",
            "paged_decode_attention_groups", "pkv_allocator_create",
            "pkv_allocator_destroy", "pkv_allocator_begin", "pkv_allocator_find_cached_prefix",
            "pkv_allocator_reserve", "pkv_allocator_publish", "pkv_allocator_expire",
            "pkv_allocator_release",
            "pkv_allocator_table", "pkv_allocator_refcount", "pkv_allocator_stats"]


class PkvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {_lib.pkv_status_string(code).decode()} (status {code})")
        self.code = code


def _check(fn: str, code: int) -> None:
    if code != PKV_OK:
        raise PkvError(fn, code)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return PKV_F32
    if t == torch.bfloat16:
        return PKV_BF16
    if t == torch.uint8:
        return PKV_FP8_E4M3
    raise TypeError(f"unsupported dtype {t}: the pools hold float32, bfloat16 or FP8 (uint8) codes")


def _act_dtype(pool_dtype: torch.dtype) -> torch.dtype:
    """dtype of queries, outputs and new rows for a pool: bf16 beside FP8 pools."""
    return torch.bfloat16 if pool_dtype == torch.uint8 else pool_dtype


FP8_BLOCK_SIZE = 16


def fp8_pools(num_blocks: int, num_kv_heads: int, head_dim: int, device) -> Tuple[torch.Tensor, torch.Tensor]:
    """A pair of FP8 (E4M3) pools: uint8 tile bytes [num_blocks, num_kv_heads,
    16 * head_dim] (block size 16, tile bytes in the library's fragment order)."""
    shape = (num_blocks, num_kv_heads, FP8_BLOCK_SIZE * head_dim)
    return (torch.zeros(shape, dtype=torch.uint8, device=device),
            torch.zeros(shape, dtype=torch.uint8, device=device))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _on(device: torch.device):
    """Make `device` current for a library call (the library plans for, and
    takes scratch from, the current device); a no-op when it already is."""
    if device.index is None or torch.cuda.current_device() == device.index:
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _pool(k_pool: torch.Tensor, v_pool: torch.Tensor, k_scale: Optional[float] = None,
          v_scale: Optional[float] = None) -> _Pool:
    _require(k_pool.dtype == v_pool.dtype and k_pool.shape == v_pool.shape,
             "K and V pools share a dtype and a shape")
    _require(k_pool.is_cuda and v_pool.is_cuda, "pools live on the GPU")
    _require(k_pool.is_contiguous() and v_pool.is_contiguous(), "pools are contiguous")
    if k_pool.dtype == torch.uint8:
        _require(k_pool.dim() == 3 and k_pool.shape[2] % FP8_BLOCK_SIZE == 0,
                 "FP8 pools are [num_blocks, num_kv_heads, 16 * head_dim] uint8")
        _require(k_scale is not None and v_scale is not None, "FP8 pools need k_scale and v_scale")
        nb, hkv, n = k_pool.shape
        return _Pool(k_pool.data_ptr(), v_pool.data_ptr(), nb, FP8_BLOCK_SIZE, hkv,
                     n // FP8_BLOCK_SIZE, PKV_FP8_E4M3, float(k_scale), float(v_scale))
    _require(k_pool.dim() == 4, "pools are [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_pool.shape
    return _Pool(k_pool.data_ptr(), v_pool.data_ptr(), nb, bs, hkv, d, _dtype_code(k_pool.dtype),
                 0.0, 0.0)


def _on_device(t: Optional[torch.Tensor], name: str, device) -> None:
    """Buffers the kernels read or write must live on the pools' GPU: the
    pointer of a host tensor, or of another GPU's, would be dereferenced by
    the kernel."""
    if t is not None:
        _require(t.is_cuda and t.device == device, f"{name} lives on {device}")


def _status_ok(status: Optional[torch.Tensor], device) -> None:
    if status is not None:
        _on_device(status, "status", device)
        _require(status.dtype == torch.int32 and status.numel() >= 1, "status is an int32 word")


def _i32_dev(t: torch.Tensor, name: str, device) -> torch.Tensor:
    _require(t.dtype == torch.int32 and t.is_contiguous() and t.device == device,
             f"{name} is a contiguous int32 tensor on {device}")
    return t


@dataclass
class PrefixDesc:
    """Shared-prefix descriptor: device arrays plus the host-side bounds."""
    num_groups: int
    max_group_rows: int
    max_prefix_blocks: int
    group_of_row: torch.Tensor   # int32 [batch] on the device
    prefix_blocks: torch.Tensor  # int32 [num_groups] (at least 1 element) on the device

    def _c(self) -> _Prefix:
        return _Prefix(self.num_groups, self.max_group_rows, self.max_prefix_blocks,
                       self.group_of_row.data_ptr(), self.prefix_blocks.data_ptr())


def _prefix_ok(prefix: Optional[PrefixDesc], device) -> None:
    if prefix is not None:
        _i32_dev(prefix.group_of_row, "prefix.group_of_row", device)
        _i32_dev(prefix.prefix_blocks, "prefix.prefix_blocks", device)


def prefix_groups_host(block_tables: np.ndarray, seq_lens: np.ndarray,
                       block_size: int) -> Tuple[np.ndarray, np.ndarray]:
    """Shared-prefix groups of host block tables (library helper)."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = t.shape[0]
    gor = np.empty(B, dtype=np.int32)
    pb = np.zeros(max(B, 1), dtype=np.int32)
    n = _lib.pkv_prefix_groups_host(t.ctypes.data, t.shape[1], sl.ctypes.data, B, block_size,
                                    gor.ctypes.data, pb.ctypes.data)
    if n < 0:
        raise ValueError("pkv_prefix_groups_host: invalid arguments")
    return gor, pb[:n].copy()


def make_prefix_desc(block_tables: np.ndarray, seq_lens: np.ndarray, block_size: int,
                     device) -> Optional[PrefixDesc]:
    """Derive the groups on the host and upload them; None when no rows share."""
    gor, pb = prefix_groups_host(block_tables, seq_lens, block_size)
    if len(pb) == 0:
        return None
    counts = np.bincount(gor[gor >= 0], minlength=len(pb))
    return PrefixDesc(len(pb), int(counts.max()), int(pb.max()),
                      torch.from_numpy(gor).to(device), torch.from_numpy(pb).to(device))


def slot_mapping_host(block_tables: np.ndarray, num_blocks: int, rows: np.ndarray,
                      positions: np.ndarray, block_size: int) -> np.ndarray:
    """slot = table[row][pos // bs] * bs + pos % bs (library helper); raises on a missing entry."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    r = np.ascontiguousarray(rows, dtype=np.int32)
    p = np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty(r.shape[0], dtype=np.int32)
    code = _lib.pkv_slot_mapping_host(t.ctypes.data, t.shape[1], t.shape[0], num_blocks,
                                      r.ctypes.data, p.ctypes.data, r.shape[0], block_size,
                                      out.ctypes.data)
    _check("pkv_slot_mapping_host", code)
    return out


def check_slot_mapping(slots: np.ndarray, num_blocks: int, block_size: int) -> None:
    """Debug check before an append (library helper, host arrays): every slot
    >= 0 inside the pool and no slot named by two tokens (their stores would
    race).  Raises ValueError naming the first token at fault."""
    s = np.ascontiguousarray(slots, dtype=np.int32)
    bad = ctypes.c_int32(-1)
    code = _lib.pkv_slot_mapping_check_host(s.ctypes.data, s.shape[0], num_blocks, block_size,
                                            ctypes.byref(bad))
    if code != PKV_OK:
        if bad.value < 0:
            raise ValueError("check_slot_mapping: invalid arguments")
        slot = int(s[bad.value])
        what = "lies past the pool" if slot >= num_blocks * block_size else "repeats an earlier token's"
        raise ValueError(f"check_slot_mapping: token {bad.value}'s slot {slot} {what}")


def paged_kv_append(k_pool: torch.Tensor, v_pool: torch.Tensor, slot_mapping: torch.Tensor,
                    k_new: torch.Tensor, v_new: torch.Tensor,
                    status: Optional[torch.Tensor] = None, k_scale: Optional[float] = None,
                    v_scale: Optional[float] = None) -> None:
    """Write ``k_new``/``v_new`` [T, Hkv, D] into the pools at ``slot_mapping`` [T]
    (quantized with ``k_scale``/``v_scale`` into FP8 pools)."""
    pool = _pool(k_pool, v_pool, k_scale, v_scale)
    dev = k_pool.device
    _i32_dev(slot_mapping, "slot_mapping", dev)
    _require(k_new.shape == v_new.shape and k_new.dim() == 3 and
             k_new.shape[1:] == (pool.num_kv_heads, pool.head_dim),
             "k_new/v_new are [T, num_kv_heads, head_dim]")
    act = _act_dtype(k_pool.dtype)
    _require(k_new.dtype == act and v_new.dtype == act, "new rows match the pool dtype (bf16 for FP8)")
    _require(k_new.is_contiguous() and v_new.is_contiguous(), "new rows are contiguous")
    _require(slot_mapping.dim() == 1 and slot_mapping.shape[0] == k_new.shape[0],
             "one slot per new token")
    _on_device(k_new, "k_new", dev)
    _on_device(v_new, "v_new", dev)
    _status_ok(status, dev)
    with _on(dev):
        _check("paged_kv_append", _lib.paged_kv_append(
            ctypes.byref(pool), slot_mapping.data_ptr(), k_new.shape[0], k_new.data_ptr(),
            v_new.data_ptr(), _ptr(status), _stream(dev)))


def decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          block_size: int, max_seq_len: int, window: int = 0,
                          prefix: Optional[PrefixDesc] = None) -> int:
    px = ctypes.byref(prefix._c()) if prefix is not None else None
    return int(_lib.paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                block_size, max_seq_len, window, px))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte-aligned device buffer (torch allocations are)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def paged_decode_attention(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor, window: int,
                           scale: float, out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None,
                           max_seq_len: Optional[int] = None,
                           prefix: Optional[PrefixDesc] = None,
                           status: Optional[torch.Tensor] = None,
                           k_scale: Optional[float] = None,
                           v_scale: Optional[float] = None) -> torch.Tensor:
    """Batched paged decode attention; returns ``out`` [B, Hq, D].

    ``max_seq_len`` is a host bound on ``seq_lens`` (default: the block-table
    capacity); ``workspace`` defaults to a fresh buffer of the queried size.
    FP8 pools (uint8) take bf16 queries and their ``k_scale``/``v_scale``.
    """
    pool = _pool(k_pool, v_pool, k_scale, v_scale)
    dev = k_pool.device
    _require(q.dim() == 3 and q.shape[2] == pool.head_dim and q.dtype == _act_dtype(k_pool.dtype) and
             q.is_contiguous() and q.device == dev, "q is [B, Hq, D], contiguous, pool dtype")
    B, hq, D = q.shape
    _i32_dev(block_tables, "block_tables", dev)
    _i32_dev(seq_lens, "seq_lens", dev)
    _require(block_tables.dim() == 2 and block_tables.shape[0] == B and seq_lens.shape == (B,),
             "block_tables [B, max_blocks], seq_lens [B]")
    width = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = width * pool.block_size
    if out is None:
        out = torch.empty_like(q)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out matches q")
    _on_device(out, "out", dev)
    _on_device(workspace, "workspace", dev)
    _status_ok(status, dev)
    _prefix_ok(prefix, dev)
    with _on(dev):  # the plan reads the SM count of the current device
        need = decode_workspace_size(B, hq, pool.num_kv_heads, D, pool.block_size, max_seq_len,
                                     window, prefix)
        if workspace is None:
            workspace = alloc_workspace(need, dev)
        px = ctypes.byref(prefix._c()) if prefix is not None else None
        _check("paged_decode_attention", _lib.paged_decode_attention(
            q.data_ptr(), hq, ctypes.byref(pool), block_tables.data_ptr(), width,
            seq_lens.data_ptr(), B, max_seq_len, window, float(scale), out.data_ptr(),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(), px, _ptr(status),
            _stream(dev)))
    return out


def prefill_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           block_size: int, max_q_len: int, max_seq_len: int,
                           window: int = 0) -> int:
    return int(_lib.paged_prefill_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_q_len, max_seq_len, window))


def paged_prefill_chunk_attention(q: torch.Tensor, cu_q_lens: torch.Tensor, k_pool: torch.Tensor,
                                  v_pool: torch.Tensor, block_tables: torch.Tensor,
                                  seq_lens: torch.Tensor, max_q_len: int, window: int,
                                  scale: float, out: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None,
                                  max_seq_len: Optional[int] = None,
                                  status: Optional[torch.Tensor] = None,
                                  k_scale: Optional[float] = None,
                                  v_scale: Optional[float] = None) -> torch.Tensor:
    """Chunked prefill against the paged prefix; returns ``out`` [sum C, Hq, D]."""
    pool = _pool(k_pool, v_pool, k_scale, v_scale)
    dev = k_pool.device
    _require(q.dim() == 3 and q.shape[2] == pool.head_dim and q.dtype == _act_dtype(k_pool.dtype) and
             q.is_contiguous() and q.device == dev, "q is [sum C, Hq, D], contiguous, pool dtype")
    _i32_dev(cu_q_lens, "cu_q_lens", dev)
    _i32_dev(block_tables, "block_tables", dev)
    _i32_dev(seq_lens, "seq_lens", dev)
    B = seq_lens.shape[0]
    _require(cu_q_lens.shape == (B + 1,) and block_tables.shape[0] == B,
             "cu_q_lens [B+1], block_tables [B, max_blocks]")
    width = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = width * pool.block_size
    if out is None:
        out = torch.empty_like(q)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out matches q")
    _on_device(out, "out", dev)
    _on_device(workspace, "workspace", dev)
    _status_ok(status, dev)
    hq = q.shape[1]
    with _on(dev):  # the plan reads the SM count of the current device
        need = prefill_workspace_size(B, hq, pool.num_kv_heads, pool.head_dim, pool.block_size,
                                      max_q_len, max_seq_len, window)
        if workspace is None:
            workspace = alloc_workspace(need, dev)
        _check("paged_prefill_chunk_attention", _lib.paged_prefill_chunk_attention(
            q.data_ptr(), cu_q_lens.data_ptr(), hq, ctypes.byref(pool), block_tables.data_ptr(),
            width, seq_lens.data_ptr(), B, max_q_len, max_seq_len, window, float(scale),
            out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _ptr(status), _stream(dev)))
    return out


def set_decode_split_blocks(n: int) -> int:
    """Diagnostic split-size override (0 = automatic); returns the previous value."""
    return int(_lib.pkv_set_decode_split_blocks(n))


def decode_plan(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                max_seq_len: int, window: int = 0) -> Tuple[int, int]:
    """(splits per row, blocks per split) of the automatic plan on the current device."""
    c = ctypes.c_int32(0)
    n = _lib.pkv_decode_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                             window, ctypes.byref(c))
    return int(n), int(c.value)


def version() -> str:
    return _lib.pkv_version().decode()


def profile_enable(kinds=()) -> None:
    """Time every launch of the given kernel kinds with CUDA events on its stream."""
    mask = 0
    for k in kinds:
        mask |= 1 << k
    _check("pkv_profile_enable", _lib.pkv_profile_enable(mask))


def profile_mask(kinds=()) -> None:
    """Change which kernel kinds are timed, keeping the records so far."""
    mask = 0
    for k in kinds:
        mask |= 1 << k
    _check("pkv_profile_mask", _lib.pkv_profile_mask(mask))


def profile_read(kind: int) -> Tuple[int, float]:
    """(launches, summed device milliseconds) recorded for a kernel kind."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check("pkv_profile_read", _lib.pkv_profile_read(kind, ctypes.byref(n), ctypes.byref(ms)))
    return int(n.value), float(ms.value)


def profile_times(kind: int) -> list:
    """Device milliseconds of every recorded launch of a kernel kind, in launch order."""
    n = ctypes.c_int64(0)
    _check("pkv_profile_times", _lib.pkv_profile_times(kind, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_float * max(int(n.value), 1))()
    _check("pkv_profile_times", _lib.pkv_profile_times(kind, buf, int(n.value), ctypes.byref(n)))
    return [float(buf[i]) for i in range(int(n.value))]


DRILL_WITHHOLD_FIRST_LOAD = 1


def set_wait_drill(wait_limit_ns: int = 0, flags: int = 0) -> None:
    """Diagnostic fail-closed drill for the launches that follow: the limit of
    each pipeline data wait (0 = the 2 s default) and, with
    DRILL_WITHHOLD_FIRST_LOAD, every pipeline's first load left unissued so
    that the wait for it runs out.  set_wait_drill() restores normal operation."""
    _check("pkv_set_wait_drill", _lib.pkv_set_wait_drill(int(wait_limit_ns), int(flags)))


def launch_count() -> int:
    """Kernels launched through the library by this process."""
    return int(_lib.pkv_launch_count())


@dataclass
class DecodeGroup:
    """One group of a fused decode: a paged_decode_attention call's own
    arguments (q [B, Hq, D], pools, tables, lengths, window, scale)."""
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    window: int
    scale: float
    out: Optional[torch.Tensor] = None
    max_seq_len: Optional[int] = None
    k_scale: Optional[float] = None
    v_scale: Optional[float] = None


def _group_c(g: DecodeGroup) -> _Group:
    pool = _pool(g.k_pool, g.v_pool, g.k_scale, g.v_scale)
    dev = g.k_pool.device
    _require(g.q.dim() == 3 and g.q.shape[2] == pool.head_dim and
             g.q.dtype == _act_dtype(g.k_pool.dtype) and g.q.is_contiguous() and g.q.device == dev,
             "q is [B, Hq, D], contiguous, pool dtype")
    B = g.q.shape[0]
    _i32_dev(g.block_tables, "block_tables", dev)
    _i32_dev(g.seq_lens, "seq_lens", dev)
    _require(g.block_tables.dim() == 2 and g.block_tables.shape[0] == B and g.seq_lens.shape == (B,),
             "block_tables [B, max_blocks], seq_lens [B]")
    if g.out is None:
        g.out = torch.empty_like(g.q)
    _require(g.out.shape == g.q.shape and g.out.dtype == g.q.dtype and g.out.is_contiguous(),
             "out matches q")
    _on_device(g.out, "out", dev)
    width = g.block_tables.shape[1]
    msl = g.max_seq_len if g.max_seq_len is not None else width * pool.block_size
    return _Group(g.q.data_ptr(), g.out.data_ptr(), pool, g.block_tables.data_ptr(), width,
                  g.seq_lens.data_ptr(), msl, int(g.window), float(g.scale))


def paged_decode_attention_groups(groups, workspace: Optional[torch.Tensor] = None,
                                  status: Optional[torch.Tensor] = None):
    """Several decode calls (groups of layers sharing the head shape: a full
    group and a sliding group, say) in one split launch and one merge launch.
    Returns the groups' outputs; each equals its own paged_decode_attention
    call bit for bit."""
    groups = list(groups)
    _require(1 <= len(groups) <= MAX_DECODE_GROUPS, f"1 .. {MAX_DECODE_GROUPS} groups")
    arr = (_Group * len(groups))(*[_group_c(g) for g in groups])
    B, hq = groups[0].q.shape[0], groups[0].q.shape[1]
    _require(all(g.q.shape[:2] == (B, hq) for g in groups), "every group has the same batch and q heads")
    dev = groups[0].k_pool.device
    _require(all(g.k_pool.device == dev for g in groups), "every group's pools on one GPU")
    _on_device(workspace, "workspace", dev)
    _status_ok(status, dev)
    with _on(dev):  # the plan reads the SM count of the current device
        need = int(_lib.paged_decode_groups_workspace_size(arr, len(groups), B, hq))
        if workspace is None:
            workspace = alloc_workspace(need, dev)
        _check("paged_decode_attention_groups", _lib.paged_decode_attention_groups(
            arr, len(groups), B, hq, workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _ptr(status), _stream(dev)))
    return [g.out for g in groups]


def decode_groups_workspace_size(groups) -> int:
    groups = list(groups)
    arr = (_Group * len(groups))(*[_group_c(g) for g in groups])
    return int(_lib.paged_decode_groups_workspace_size(arr, len(groups), groups[0].q.shape[0],
                                                       groups[0].q.shape[1]))


def paged_decode_attention_no_alloc(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                    block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                    window: int, scale: float, out: torch.Tensor,
                                    max_seq_len: Optional[int] = None,
                                    prefix: Optional[PrefixDesc] = None,
                                    status: Optional[torch.Tensor] = None,
                                    k_scale: Optional[float] = None,
                                    v_scale: Optional[float] = None) -> torch.Tensor:
    """paged_decode_attention for callers that cannot allocate device memory.

    No workspace is passed and nothing is allocated: the library's fixed
    device scratch (``NO_ALLOC_SCRATCH_BYTES`` per GPU) is used, and ``out``
    must be given.  Calls on one device share that scratch, so calls that may
    overlap on the GPU must be ordered.  Sizes that need more scratch raise
    PkvError with PKV_ERR_WORKSPACE.
    """
    pool = _pool(k_pool, v_pool, k_scale, v_scale)
    dev = k_pool.device
    _require(q.dim() == 3 and q.shape[2] == pool.head_dim and q.dtype == _act_dtype(k_pool.dtype) and
             q.is_contiguous() and q.device == dev, "q is [B, Hq, D], contiguous, pool dtype")
    B, hq, _ = q.shape
    _i32_dev(block_tables, "block_tables", dev)
    _i32_dev(seq_lens, "seq_lens", dev)
    _require(block_tables.dim() == 2 and block_tables.shape[0] == B and seq_lens.shape == (B,),
             "block_tables [B, max_blocks], seq_lens [B]")
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out matches q")
    _on_device(out, "out", dev)
    _status_ok(status, dev)
    _prefix_ok(prefix, dev)
    width = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = width * pool.block_size
    px = ctypes.byref(prefix._c()) if prefix is not None else None
    # the pools' GPU is made current for the call: the library takes the
    # scratch of the current device and launches on this device's stream
    with _on(dev):
        code = _lib.paged_decode_attention_no_alloc(
            q.data_ptr(), hq, ctypes.byref(pool), block_tables.data_ptr(), width,
            seq_lens.data_ptr(), B, max_seq_len, window, float(scale), out.data_ptr(), px,
            _ptr(status), _stream(dev))
    if code == PKV_ERR_WORKSPACE:
        raise PkvError("paged_decode_attention_no_alloc (request exceeds the "
                       f"{NO_ALLOC_SCRATCH_BYTES >> 20} MiB static scratch)", code)
    _check("paged_decode_attention_no_alloc", code)
    return out


# ---------------------------------------------------------------------------
# host block allocator
# ---------------------------------------------------------------------------
class BlockAllocator:
    """The library's host block allocator (see ``include/pkv.h``): block ids of
    a pool of ``block_size``-token blocks, shared across requests by prefix
    hash, refcounted, with LRU eviction of cache-only blocks and
    grow-on-demand up to ``max_blocks``.  Token lists are int32 sequences."""

    def __init__(self, block_size: int, initial_blocks: int, max_blocks: int):
        self._a = _lib.pkv_allocator_create(block_size, initial_blocks, max_blocks)
        _require(bool(self._a), "block_size > 0 and 0 <= initial_blocks <= max_blocks")
        self.block_size = block_size

    def __del__(self):
        a = getattr(self, "_a", None)
        if a:
            _lib.pkv_allocator_destroy(a)
            self._a = None

    @staticmethod
    def _tokens(tokens):
        arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return arr, (arr.ctypes.data if arr.size else None)

    @staticmethod
    def _keys(extra_keys):
        if extra_keys is None:
            return None, None
        arr = np.ascontiguousarray(np.asarray(extra_keys, dtype=np.uint64))
        return arr, arr.ctypes.data

    def begin(self) -> int:
        return int(_lib.pkv_allocator_begin(self._a))

    def find_cached_prefix(self, req: int, tokens, extra_keys=None) -> int:
        t, tp = self._tokens(tokens)
        k, kp = self._keys(extra_keys)
        n = ctypes.c_int32(0)
        _check("pkv_allocator_find_cached_prefix",
               _lib.pkv_allocator_find_cached_prefix(self._a, req, tp, t.size, kp, ctypes.byref(n)))
        return int(n.value)

    def reserve(self, req: int, n_tokens: int) -> None:
        _check("pkv_allocator_reserve", _lib.pkv_allocator_reserve(self._a, req, int(n_tokens)))

    def publish(self, req: int, tokens, extra_keys=None) -> None:
        t, tp = self._tokens(tokens)
        k, kp = self._keys(extra_keys)
        _check("pkv_allocator_publish", _lib.pkv_allocator_publish(self._a, req, tp, t.size, kp))

    def expire(self, req: int, first_live_token: int) -> None:
        """Drop the blocks wholly before ``first_live_token`` (a sliding
        window's start); their table entries become -1."""
        _check("pkv_allocator_expire", _lib.pkv_allocator_expire(self._a, req, int(first_live_token)))

    def release(self, req: int) -> None:
        _check("pkv_allocator_release", _lib.pkv_allocator_release(self._a, req))

    def table(self, req: int) -> np.ndarray:
        n = ctypes.c_int32(0)
        _check("pkv_allocator_table", _lib.pkv_allocator_table(self._a, req, None, 0, ctypes.byref(n)))
        out = np.empty(n.value, dtype=np.int32)
        if n.value:
            _check("pkv_allocator_table", _lib.pkv_allocator_table(
                self._a, req, out.ctypes.data, n.value, ctypes.byref(n)))
        return out

    def refcount(self, block: int) -> int:
        return int(_lib.pkv_allocator_refcount(self._a, block))

    def stats(self):
        """(num_blocks, free_blocks, cached_blocks, grows)."""
        v = [ctypes.c_int32(0) for _ in range(4)]
        _check("pkv_allocator_stats", _lib.pkv_allocator_stats(self._a, *[ctypes.byref(x) for x in v]))
        return tuple(int(x.value) for x in v)
