"""The C-ABI library on the CPU: it loads, exports every function that
include/pkv.h declares, its host helpers agree bit for bit with the oracle's
independent derivations, and argument checks fail before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import pkv_inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def pkv():
    import block_paged_kv_gb300 as m
    return m


def test_header_symbols_exported(pkv):
    names = declared_functions()
    assert "paged_kv_append" in names and "paged_decode_attention" in names
    lib = ctypes.CDLL(pkv.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(pkv.EXPORTED) <= set(names)


def _workloads():
    return [gen.tiny_f32(), gen.dense_bf16(), gen.shared_prefix_b32(batch=8, max_suffix=200),
            *gen.long_two_groups(batch=2, context=512, window=64),
            gen.chunked_prefill(batch=2, chunk=40, prefix=64)]


def test_slot_mapping_matches_oracle(pkv, orc):
    for w in _workloads():
        lib_slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                          w.block_size)
        or_slots, bad = orc.slot_mapping(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                         w.block_size)
        assert bad == 0 and np.array_equal(lib_slots, or_slots), w.name


def test_slot_mapping_rejects_missing_entry(pkv):
    t = np.array([[3, -1]], dtype=np.int32)
    with pytest.raises(pkv.PkvError):
        pkv.slot_mapping_host(t, 8, np.array([0], np.int32), np.array([20], np.int32), 16)


def test_prefix_groups_match_oracle(pkv, orc):
    for w in _workloads():
        a = pkv.prefix_groups_host(w.block_tables, w.seq_lens, w.block_size)
        b = orc.prefix_groups(w.block_tables, w.seq_lens, w.block_size)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), w.name
    w = gen.shared_prefix_b32(batch=8, max_suffix=200)
    gor, pb = pkv.prefix_groups_host(w.block_tables, w.seq_lens, 16)
    assert gor.tolist() == [0] * 8 and pb.tolist() == [64]
    for seed in range(20):
        u = gen.uniform_ints(900 + seed, "t", 30 * 5, -1, 6).reshape(30, 5).astype(np.int32)
        L = gen.uniform_ints(950 + seed, "l", 30, -3, 90).astype(np.int32)
        a = pkv.prefix_groups_host(u, L, 16)
        b = orc.prefix_groups(u, L, 16)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), seed


def test_argument_checks_before_launch(pkv):
    lib = pkv._lib
    # null pool
    assert lib.paged_kv_append(None, None, 1, None, None, None, None) == pkv.PKV_ERR_INVALID_ARG
    pool = pkv._Pool(16, 16, 4, 16, 2, 64, pkv.PKV_BF16)
    # misaligned new rows
    assert lib.paged_kv_append(ctypes.byref(pool), 16, 1, 8, 16, None, None) == pkv.PKV_ERR_INVALID_ARG
    # head_dim not divisible by the kv heads' query groups
    assert lib.paged_decode_attention(16, 3, ctypes.byref(pool), 16, 4, 16, 1, 64, 0, 1.0, 16, 256,
                                      1 << 20, None, None, None) == pkv.PKV_ERR_INVALID_ARG
    # negative window
    assert lib.paged_decode_attention(16, 4, ctypes.byref(pool), 16, 4, 16, 1, 64, -1, 1.0, 16, 256,
                                      1 << 20, None, None, None) == pkv.PKV_ERR_INVALID_ARG
    # bf16 with a block size the bf16 kernel is not built for
    pool32 = pkv._Pool(16, 16, 4, 32, 2, 64, pkv.PKV_BF16)
    assert lib.paged_decode_attention(16, 4, ctypes.byref(pool32), 16, 4, 16, 1, 64, 0, 1.0, 16,
                                      256, 1 << 20, None, None, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_status_string(pkv.PKV_ERR_WORKSPACE).decode() == "workspace too small or misaligned"


def test_plain_c_caller(pkv, tmp_path):
    """include/pkv.h compiles as C99 and a C program linked against the library
    runs its host-side entry points (tests/c_abi_host.c) without torch."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    libdir = os.path.dirname(pkv.LIB_PATH)
    exe = str(tmp_path / "c_abi_host")
    build = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror",
                            "-I", os.path.join(ROOT, "include"),
                            os.path.join(ROOT, "tests", "c_abi_host.c"),
                            "-L", libdir, "-lpkv", f"-Wl,-rpath,{libdir}", "-o", exe],
                           capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    assert "c_abi_host: ok" in run.stdout


def _first_fault(slots, cap):
    seen = set()
    for i, s in enumerate(int(x) for x in slots):
        if s < 0:
            continue
        if s >= cap or s in seen:
            return i
        seen.add(s)
    return None


def test_slot_mapping_check(pkv):
    # the appends of the workloads: slots inside the pool, none repeated
    for w in _workloads():
        slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                      w.block_size)
        pkv.check_slot_mapping(slots, w.num_blocks, w.block_size)
    # seeded slot arrays with planted repeats and out-of-pool slots: the first
    # token at fault, in order, is the one named
    nb, bs = 8, 16
    for seed in range(40):
        s = gen.uniform_ints(700 + seed, "slots", 24, -2, nb * bs + 3).astype(np.int32)
        want = _first_fault(s, nb * bs)
        if want is None:
            pkv.check_slot_mapping(s, nb, bs)
            continue
        with pytest.raises(ValueError, match=f"token {want}'s slot {int(s[want])} "):
            pkv.check_slot_mapping(s, nb, bs)
    # negative slots are skipped by the append, so they may repeat
    pkv.check_slot_mapping(np.array([-1, 5, -1, 6], np.int32), nb, bs)
    with pytest.raises(ValueError, match="token 2's slot 5 repeats"):
        pkv.check_slot_mapping(np.array([5, 7, 5], np.int32), nb, bs)
    with pytest.raises(ValueError, match="past the pool"):
        pkv.check_slot_mapping(np.array([3, nb * bs], np.int32), nb, bs)
    with pytest.raises(ValueError, match="invalid arguments"):
        pkv.check_slot_mapping(np.array([3], np.int32), 0, bs)
