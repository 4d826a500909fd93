"""CPU oracle for the block-paged KV attention path (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does, and this
package imports nothing from the library.

The arithmetic lives in ``pkv_oracle.c`` (plain loops, IEEE double on exactly
widened float32/bf16 inputs and exactly decoded E4M3 codes); this file
compiles it with gcc and marshals numpy arrays through ctypes.  Every
attention function returns float64 outputs.

Parity status: every oracle function is pinned by ``tests/test_oracle_pins.py``
(closed forms, library dense attention on gathered keys, 50-digit brute force,
invariances, a golden fixture and planted-mistake checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")

DTYPE_CODE = {"f32": 0, "bf16": 1, "fp8": 2}
FP8_BLOCK = 16   # tokens per block of an FP8 pool

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_dbl = ctypes.c_double
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


def build(out_path: str = _LIB_PATH, defines: Sequence[str] = (), force: bool = False) -> str:
    """Compile the oracle (``-O2``, no fast-math: IEEE semantics kept)."""
    if not force and os.path.exists(out_path) and not defines \
            and os.path.getmtime(out_path) >= os.path.getmtime(_SRC):
        return out_path
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
           *[f"-D{d}" for d in defines], _SRC, "-o", out_path + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out_path + ".tmp", out_path)
    return out_path


class Oracle:
    """ctypes view of one compiled oracle (the normal build or a planted variant)."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.or_slot_mapping.argtypes = [_i32p, _i32, _i32, _i32, _i32p, _i32p, _i32, _i32, _i32p]
        lib.or_slot_mapping.restype = _i32
        lib.or_append.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32p, _i32, _vp, _vp,
                                  ctypes.c_float, ctypes.c_float]
        lib.or_append.restype = _i32
        lib.or_decode.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32p, _i32,
                                  _i32p, _i32, _i32, _dbl, _dbl, _dbl, _f64p]
        lib.or_decode.restype = _i32
        lib.or_decode_pairs.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32p,
                                        _i32, _i32p, _i32, _dbl, _dbl, _dbl, _i32p, _i32p, _i32,
                                        _f64p]
        lib.or_decode_pairs.restype = _i32
        lib.or_prefill.argtypes = [_vp, _i32p, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                   _i32p, _i32, _i32p, _i32, _i32, _dbl, _dbl, _dbl, _f64p]
        lib.or_prefill.restype = _i32
        lib.or_prefill_samples.argtypes = [_vp, _i32p, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                           _i32, _i32p, _i32, _i32p, _i32, _dbl, _dbl, _dbl,
                                           _i32p, _i32p, _i32p, _i32, _f64p]
        lib.or_prefill_samples.restype = _i32
        lib.or_prefix_groups.argtypes = [_i32p, _i32, _i32p, _i32, _i32, _i32p, _i32p]
        lib.or_prefix_groups.restype = _i32
        lib.or_e4m3_decode.argtypes = [_u8p, _i32, _f64p]
        lib.or_e4m3_decode.restype = None
        lib.or_e4m3_encode.argtypes = [_f32p, _i32, _u8p]
        lib.or_e4m3_encode.restype = None
        self.lib = lib

    # -- helpers -------------------------------------------------------------
    @staticmethod
    def _c(a: np.ndarray, dtype=None) -> np.ndarray:
        return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))

    @staticmethod
    def _ptr(a: np.ndarray) -> int:
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data

    @staticmethod
    def _pool_shape(pool: np.ndarray, dtype: str):
        """(num_blocks, Hkv, block_size, head_dim) of a pool array: [nb, Hkv, bs, D],
        or for FP8 the tile bytes [nb, Hkv, 16 * D] (uint8)."""
        if dtype == "fp8":
            nb, hkv, n = pool.shape
            assert pool.dtype == np.uint8 and n % FP8_BLOCK == 0
            return nb, hkv, FP8_BLOCK, n // FP8_BLOCK
        return pool.shape

    # -- E4M3 codec (pins) ---------------------------------------------------
    def e4m3_decode(self, codes: np.ndarray) -> np.ndarray:
        c = self._c(codes, np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.or_e4m3_decode(c.reshape(-1), c.size, out.reshape(-1))
        return out

    def e4m3_encode(self, x: np.ndarray) -> np.ndarray:
        x = self._c(x, np.float32)
        out = np.empty(x.shape, dtype=np.uint8)
        self.lib.or_e4m3_encode(x.reshape(-1), x.size, out.reshape(-1))
        return out

    # -- slot mapping --------------------------------------------------------
    def slot_mapping(self, tables: np.ndarray, num_blocks: int, rows: np.ndarray,
                     pos: np.ndarray, block_size: int):
        t = self._c(tables, np.int32)
        rows = self._c(rows, np.int32)
        pos = self._c(pos, np.int32)
        out = np.empty(rows.shape[0], dtype=np.int32)
        bad = self.lib.or_slot_mapping(t, t.shape[1], t.shape[0], num_blocks, rows, pos,
                                       rows.shape[0], block_size, out)
        return out, int(bad)

    # -- append (in place on the given pools) --------------------------------
    def append(self, k_pool: np.ndarray, v_pool: np.ndarray, dtype: str, slots: np.ndarray,
               k_new: np.ndarray, v_new: np.ndarray, k_scale: float = 1.0,
               v_scale: float = 1.0) -> int:
        """In place.  FP8 pools take bf16 new rows (uint16 bits) and their scales."""
        assert k_pool.flags["C_CONTIGUOUS"] and v_pool.flags["C_CONTIGUOUS"]
        nb, hkv, bs, d = self._pool_shape(k_pool, dtype)
        slots = self._c(slots, np.int32)
        kn, vn = self._c(k_new), self._c(v_new)
        if dtype == "fp8":
            assert kn.dtype == np.uint16 and vn.dtype == np.uint16
        bad = int(self.lib.or_append(self._ptr(k_pool), self._ptr(v_pool), DTYPE_CODE[dtype], nb,
                                     hkv, bs, d, slots, slots.shape[0], self._ptr(kn),
                                     self._ptr(vn), k_scale, v_scale))
        if bad < 0:
            raise ValueError("oracle append: an FP8 pool needs 16-token blocks and head_dim % 64 == 0")
        return bad

    # -- decode --------------------------------------------------------------
    def decode(self, q, k_pool, v_pool, dtype: str, tables, seq_lens, window: int, scale: float,
               pairs: Optional[np.ndarray] = None, k_scale: float = 1.0, v_scale: float = 1.0):
        """Full [B, Hq, D] output, or [n, D] for ``pairs`` = int array [n, 2] of (row, head).
        ``dtype`` "fp8": bf16 queries against E4M3 pools with their scales."""
        q, kp, vp = self._c(q), self._c(k_pool), self._c(v_pool)
        t = self._c(tables, np.int32)
        sl = self._c(seq_lens, np.int32)
        nb, hkv, bs, d = self._pool_shape(kp, dtype)
        hq = q.shape[1]
        if pairs is None:
            out = np.zeros((q.shape[0], hq, d), dtype=np.float64)
            bad = self.lib.or_decode(self._ptr(q), self._ptr(kp), self._ptr(vp), DTYPE_CODE[dtype],
                                     nb, hq, hkv, bs, d, t, t.shape[1], sl, sl.shape[0], window,
                                     scale, k_scale, v_scale, out)
        else:
            pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
            rows, heads = self._c(pairs[:, 0]), self._c(pairs[:, 1])
            out = np.zeros((pairs.shape[0], d), dtype=np.float64)
            bad = self.lib.or_decode_pairs(self._ptr(q), self._ptr(kp), self._ptr(vp),
                                           DTYPE_CODE[dtype], nb, hq, hkv, bs, d, t, t.shape[1],
                                           sl, window, scale, k_scale, v_scale, rows, heads,
                                           rows.shape[0], out)
        if bad < 0:
            raise ValueError("oracle decode: an FP8 pool needs 16-token blocks and head_dim % 64 == 0")
        if bad:
            raise ValueError(f"oracle decode: {bad} outputs read a missing or out-of-pool block")
        return out

    # -- prefill -------------------------------------------------------------
    def prefill(self, q, cu_q_lens, k_pool, v_pool, dtype: str, tables, seq_lens, window: int,
                scale: float, samples: Optional[np.ndarray] = None, k_scale: float = 1.0,
                v_scale: float = 1.0):
        """Full [sum C, Hq, D] output, or [n, D] for ``samples`` = [n, 3] of
        (row, query index in the row's chunk, head)."""
        q, kp, vp = self._c(q), self._c(k_pool), self._c(v_pool)
        cu = self._c(cu_q_lens, np.int32)
        t = self._c(tables, np.int32)
        sl = self._c(seq_lens, np.int32)
        nb, hkv, bs, d = self._pool_shape(kp, dtype)
        hq = q.shape[1]
        if samples is None:
            out = np.zeros((q.shape[0], hq, d), dtype=np.float64)
            bad = self.lib.or_prefill(self._ptr(q), cu, self._ptr(kp), self._ptr(vp),
                                      DTYPE_CODE[dtype], nb, hq, hkv, bs, d, t, t.shape[1], sl,
                                      sl.shape[0], window, scale, k_scale, v_scale, out)
        else:
            s = np.asarray(samples, dtype=np.int32).reshape(-1, 3)
            rows, qi, heads = self._c(s[:, 0]), self._c(s[:, 1]), self._c(s[:, 2])
            out = np.zeros((s.shape[0], d), dtype=np.float64)
            bad = self.lib.or_prefill_samples(self._ptr(q), cu, self._ptr(kp), self._ptr(vp),
                                              DTYPE_CODE[dtype], nb, hq, hkv, bs, d, t,
                                              t.shape[1], sl, window, scale, k_scale, v_scale,
                                              rows, qi, heads, rows.shape[0], out)
        if bad < 0:
            raise ValueError("oracle prefill: an FP8 pool needs 16-token blocks and head_dim % 64 == 0")
        if bad:
            raise ValueError(f"oracle prefill: {bad} outputs read a missing or out-of-pool block")
        return out

    # -- shared-prefix groups ------------------------------------------------
    def prefix_groups(self, tables, seq_lens, block_size: int):
        t = self._c(tables, np.int32)
        sl = self._c(seq_lens, np.int32)
        B = t.shape[0]
        gor = np.empty(B, dtype=np.int32)
        pb = np.zeros(max(B, 1), dtype=np.int32)
        ng = self.lib.or_prefix_groups(t, t.shape[1], sl, B, block_size, gor, pb)
        return gor, pb[:ng].copy()


_default: Optional[Oracle] = None


def load() -> Oracle:
    """The normal oracle build (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def load_planted(defines: Sequence[str]) -> Oracle:
    """An oracle compiled with planted mistakes (for the pin tests only)."""
    d = tempfile.mkdtemp(prefix="pkv_oracle_plant_")
    return Oracle(build(os.path.join(d, "liboracle_" + "_".join(defines) + ".so"), defines,
                        force=True))
