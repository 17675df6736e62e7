"""Host-side tests of the C ABI that need no GPU.

- every function declared in include/hicache.h is exported by the library;
- the run planner against brute force;
- argument and index validation, which completes before any CUDA call, so it
  can be driven with placeholder device pointers.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import hierarchical_kv_cache_gb300 as hk
from hierarchical_kv_cache_gb300 import _binding as B
from hierarchical_kv_cache_gb300.build import build

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def declared_functions():
    text = open(os.path.join(REPO, "include", "hicache.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hicache_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported():
    names = declared_functions()
    assert "hicache_backup_all_layers" in names and "hicache_load_burst" in names
    lib = ctypes.CDLL(B.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert hk.abi_version() == 5


def brute_runs(d, h, P):
    runs = []
    for i in range(len(d)):
        if runs and d[i] == runs[-1][0] + runs[-1][2] and h[i] == runs[-1][1] + runs[-1][2] \
                and h[i] % P != 0:
            runs[-1][2] += 1
        else:
            runs.append([int(d[i]), int(h[i]), 1])
    return runs


@pytest.mark.parametrize("P", [1, 2, 3, 16, 64])
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_plan_runs_matches_brute_force(P, dtype):
    g = np.random.default_rng(P)
    for trial in range(20):
        n = int(g.integers(0, 300))
        # mix of contiguous stretches and jumps
        d = np.cumsum(np.where(g.random(n) < 0.8, 1, g.integers(2, 50, n))).astype(dtype)
        h = np.cumsum(np.where(g.random(n) < 0.8, 1, g.integers(2, 50, n))).astype(dtype)
        runs, full = hk.hicache_plan_runs(d, h, P)
        want = brute_runs(d, h, P)
        assert runs.tolist() == want
        assert full == sum(1 for r in want if r[2] == P and r[1] % P == 0)
        if n:
            assert runs[:, 2].sum() == n


def test_plan_runs_whole_pages():
    P = 64
    pages = np.array([7, 3, 4, 5, 100])
    h = (pages[:, None] * P + np.arange(P)).reshape(-1)
    d = np.arange(h.size) + 640
    runs, full = hk.hicache_plan_runs(d, h, P)
    assert len(runs) == 5 and full == 5  # runs never cross a host page boundary


# ---- validation with placeholder pointers: every rejected call returns before any CUDA call

FAKE = 0x10000  # 64 KiB-aligned placeholder address, never dereferenced


def c_pool(L=2, T=2, head_num=2, head_dim=8, dtype_size=2, P=4, slots=64, pages=8,
           page_granular=0, dev_ptrs=None, host_ptrs=None, layout=0):
    dev = (ctypes.c_void_p * (T * L))(*(dev_ptrs or [FAKE + 0x100000 * i for i in range(T * L)]))
    host = (ctypes.c_void_p * T)(*(host_ptrs or [FAKE + 0x10000000 * (i + 1) for i in range(T)]))
    p = B.c_pool(num_layers=L, num_tensors=T, head_num=head_num, head_dim=head_dim,
                 dtype_size=dtype_size, page_size=P, page_granular=page_granular, layout=layout,
                 device_slots=slots, host_pages=pages,
                 device_layers=ctypes.cast(dev, ctypes.POINTER(ctypes.c_void_p)),
                 host_tensors=ctypes.cast(host, ctypes.POINTER(ctypes.c_void_p)))
    p._keep = (dev, host)
    return p


def call_backup(pools, d, h, opts=None):
    arr = (B.c_pool * len(pools))(*pools)
    d = np.ascontiguousarray(d, dtype=np.int64)
    h = np.ascontiguousarray(h, dtype=np.int64)
    o = opts or B.c_opts(path=0, index_location=0)
    return B.lib().hicache_backup_all_layers(arr, len(pools), d.ctypes.data, h.ctypes.data, 64,
                                             d.size, ctypes.byref(o), None)


def call_load(pools, layer, h, d, opts=None):
    arr = (B.c_pool * len(pools))(*pools)
    d = np.ascontiguousarray(d, dtype=np.int64)
    h = np.ascontiguousarray(h, dtype=np.int64)
    o = opts or B.c_opts(path=0, index_location=0)
    return B.lib().hicache_load_layer(arr, len(pools), layer, h.ctypes.data, d.ctypes.data, 64,
                                      d.size, ctypes.byref(o), None, None)


def err():
    return B.lib().hicache_last_error().decode()


def test_rejects_bad_pool_arguments():
    lib = B.lib()
    assert lib.hicache_backup_all_layers(None, 1, None, None, 64, 0, None, None) == B.HICACHE_EINVAL
    assert "NULL" in err()
    assert call_backup([c_pool(L=0)], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(T=3)], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(head_dim=3, dtype_size=1, head_num=1)], [], []) == B.HICACHE_EALIGN
    assert call_backup([c_pool(dev_ptrs=[FAKE + 2] * 4)], [], []) == B.HICACHE_EALIGN
    assert call_backup([c_pool(dev_ptrs=[0] * 4)], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(P=0)], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(L=2), c_pool(L=3)], [], []) == B.HICACHE_EINVAL
    assert "num_layers" in err()
    assert call_backup([c_pool(P=4), c_pool(P=8)], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(page_granular=1, slots=63)], [], []) == B.HICACHE_EINVAL
    o = B.c_opts(path=7)
    assert call_backup([c_pool()], [], [], opts=o) == B.HICACHE_EINVAL
    assert call_backup([c_pool(layout=2)], [], []) == B.HICACHE_EINVAL
    assert "layout" in err()
    assert call_backup([c_pool(layout=1)], [], []) == B.HICACHE_OK


def test_limits_are_rejected_just_beyond_the_maxima():
    assert call_backup([c_pool(L=4097)], [], []) == B.HICACHE_EINVAL  # 4096 layers at most
    assert call_backup([c_pool(L=4096)], [], []) == B.HICACHE_OK
    # rows of at most 16 MiB: 2 x 4 Mi x 2 B = 16 MiB passes, one more head does not
    assert call_backup([c_pool(head_num=2, head_dim=4 << 20, dtype_size=2)], [], []) == B.HICACHE_OK
    assert call_backup([c_pool(head_num=3, head_dim=4 << 20, dtype_size=2)], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(slots=(1 << 31))], [], []) == B.HICACHE_EINVAL
    assert call_backup([c_pool(pages=(1 << 29), P=4)], [], []) == B.HICACHE_EINVAL
    lib = B.lib()
    arr = (B.c_pool * 1)(c_pool())
    d = np.zeros(4, dtype=np.int64)
    assert lib.hicache_backup_all_layers(arr, 1, d.ctypes.data, d.ctypes.data, 64, 1 << 31, None,
                                         None) == B.HICACHE_EINVAL
    assert "2^31" in err()
    assert lib.hicache_backup_all_layers(arr, 5, d.ctypes.data, d.ctypes.data, 64, 0, None,
                                         None) == B.HICACHE_EINVAL  # at most 4 pools


def test_empty_call_is_ok_without_cuda():
    assert call_backup([c_pool()], [], []) == B.HICACHE_OK
    assert call_load([c_pool()], 1, [], []) == B.HICACHE_OK


def test_rejects_bad_index_arguments():
    lib = B.lib()
    arr = (B.c_pool * 1)(c_pool())
    d = np.zeros(4, dtype=np.int64)
    assert lib.hicache_backup_all_layers(arr, 1, d.ctypes.data, d.ctypes.data, 16, 4, None,
                                         None) == B.HICACHE_EINVAL
    assert lib.hicache_backup_all_layers(arr, 1, d.ctypes.data, None, 64, 4, None,
                                         None) == B.HICACHE_EINVAL
    assert lib.hicache_backup_all_layers(arr, 1, d.ctypes.data, d.ctypes.data, 64, -1, None,
                                         None) == B.HICACHE_EINVAL


def test_range_checks():
    pool = c_pool(slots=64, pages=8, P=4)  # host tokens 32
    assert call_backup([pool], [0, 64], [0, 1]) == B.HICACHE_ERANGE
    assert "device index 64" in err()
    assert call_backup([pool], [0, -1], [0, 1]) == B.HICACHE_ERANGE
    assert call_backup([pool], [0, 1], [0, 32]) == B.HICACHE_ERANGE
    assert "host index 32" in err()
    # the smallest pool of a call bounds the indices
    small = c_pool(slots=16, pages=8, P=4)
    assert call_backup([pool, small], [0, 20], [0, 1]) == B.HICACHE_ERANGE
    assert call_load([pool], 0, [0, 33], [1, 2]) == B.HICACHE_ERANGE


def test_duplicate_destinations():
    pool = c_pool(slots=64, pages=8, P=4)
    # backup: host destinations must be distinct, device sources may repeat
    assert call_backup([pool], [3, 4, 5], [7, 9, 7]) == B.HICACHE_EDUP
    assert "host destination 7" in err()
    # load: device destinations must be distinct, host sources may repeat
    assert call_load([pool], 0, [5, 5, 6], [1, 2, 1]) == B.HICACHE_EDUP
    assert "device destination 1" in err()
    # the duplicate bitmap is cleared between calls: a later distinct list passes validation
    # (and then fails only at the first CUDA call on a machine without a GPU)
    st = call_backup([pool], [3, 3, 3], [7, 9, 10])
    assert st in (B.HICACHE_OK, B.HICACHE_ECUDA, B.HICACHE_EINVAL)
    assert "destination" not in err()


def test_page_granular_needs_whole_pages():
    P = 4
    pool = c_pool(T=1, head_num=1, head_dim=132, dtype_size=1, P=P, slots=64, pages=8,
                  page_granular=1)
    assert call_backup([pool], [0, 1, 2], [4, 5, 6]) == B.HICACHE_EINVAL  # not a multiple of P
    assert call_backup([pool], [1, 2, 3, 4], [4, 5, 6, 7]) == B.HICACHE_EINVAL  # unaligned device
    assert call_backup([pool], [4, 5, 7, 6], [4, 5, 6, 7]) == B.HICACHE_EINVAL  # not one page
    assert "whole page" in err() or "start a page" in err()


def test_load_layer_range():
    pool = c_pool(L=2)
    assert call_load([pool], 2, [1], [1]) == B.HICACHE_EINVAL
    assert call_load([pool], -1, [1], [1]) == B.HICACHE_EINVAL
    lib = B.lib()
    arr = (B.c_pool * 1)(pool)
    assert lib.hicache_load_burst(arr, 1, 1, 3, None, None, 64, 0, None, None,
                                  None) == B.HICACHE_EINVAL


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.lib()


def test_concurrent_builds_compile_once(tmp_path):
    """Processes that build at the same time (ranks of a multi-GPU run) take turns
    on a lock: one compiles, the others find the library current and load it."""
    import subprocess
    import sys

    code = ("import time, hierarchical_kv_cache_gb300.build as b; t = time.time(); "
            "b.build(force=True); print(round(time.time() - t, 2))")
    procs = [subprocess.Popen([sys.executable, "-c", code], cwd=REPO, stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for _ in range(3)]
    outs = [p.communicate(timeout=600) for p in procs]
    assert all(p.returncode == 0 for p in procs), [o[1][-2000:] for o in outs]
    mtime = os.path.getmtime(B.LIB_PATH)
    # one build: the library is newer than every object file the others could have written
    objs = [os.path.join(os.path.dirname(B.LIB_PATH), "_build", f)
            for f in os.listdir(os.path.join(os.path.dirname(B.LIB_PATH), "_build"))
            if f.endswith(".o")]
    assert objs and all(os.path.getmtime(o) <= mtime for o in objs)
    lib = ctypes.CDLL(B.LIB_PATH)
    assert lib.hicache_abi_version() == 5
