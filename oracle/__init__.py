"""CPU oracle for the paged KV-cache transfer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never does: it has
its own CUDA path and fails loudly when that is missing.

The arithmetic lives in ``hicache_oracle.c`` (plain loops, one ``memcpy`` per
token row).  This module only compiles it (``build_oracle``), loads it and
marshals numpy arrays into its C signatures.  Index arrays of any integer
width are widened to int64 here, which is exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hicache_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_hicache.so")
_lib = None


def build_oracle(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library and return its path."""
    cmd = ["gcc", "-O1", "-std=c99", "-Wall", "-Werror", "-shared", "-fPIC",
           *extra_flags, "-o", out, src]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads another copy."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build_oracle()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.oracle_backup_all_layers.argtypes = [i64, i64, i64, i64, i64, vp, vp, vp, vp, i64]
    lib.oracle_backup_all_layers.restype = ctypes.c_int
    lib.oracle_load_layer.argtypes = [i64, i64, i64, i64, i64, i64, vp, vp, vp, vp, i64]
    lib.oracle_load_layer.restype = ctypes.c_int
    lib.oracle_load_burst.argtypes = [i64, i64, i64, i64, i64, i64, i64, vp, vp, vp, vp, i64]
    lib.oracle_load_burst.restype = ctypes.c_int
    lib.oracle_pf_backup_all_layers.argtypes = [i64, i64, i64, i64, vp, vp, vp, vp, i64]
    lib.oracle_pf_backup_all_layers.restype = ctypes.c_int
    lib.oracle_pf_load_layer.argtypes = [i64, i64, i64, i64, i64, vp, vp, vp, vp, i64]
    lib.oracle_pf_load_layer.restype = ctypes.c_int
    return lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _idx(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int64)


def _layers_array(layers):
    arr = (ctypes.c_void_p * len(layers))(*[_ptr(x) for x in layers])
    return arr


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


def backup_all_layers(device_layers, host, device_idx, host_idx, *, page_size: int,
                      row_bytes: int, lib=None) -> None:
    """Oracle all-layer backup of one tensor, in place on ``host``.

    device_layers: list of L uint8 arrays, each device_slots * row_bytes bytes.
    host: uint8 array host_pages * L * page_size * row_bytes bytes.
    """
    lib = lib or load()
    L = len(device_layers)
    for x in device_layers:
        assert x.dtype == np.uint8 and x.flags.c_contiguous
    assert host.dtype == np.uint8 and host.flags.c_contiguous
    d = _idx(device_idx)
    h = _idx(host_idx)
    assert d.shape == h.shape
    device_slots = device_layers[0].size // row_bytes
    host_pages = host.size // (L * page_size * row_bytes)
    arr = _layers_array(device_layers)
    rc = lib.oracle_backup_all_layers(L, page_size, row_bytes, device_slots, host_pages,
                                      ctypes.cast(arr, ctypes.c_void_p), _ptr(host),
                                      _ptr(d), _ptr(h), d.size)
    _check(rc, "oracle_backup_all_layers")


def load_layer(device_layer, host, layer: int, host_idx, device_idx, *, num_layers: int,
               page_size: int, row_bytes: int, lib=None) -> None:
    """Oracle load-back of one layer of one tensor, in place on ``device_layer``."""
    lib = lib or load()
    assert device_layer.dtype == np.uint8 and device_layer.flags.c_contiguous
    assert host.dtype == np.uint8 and host.flags.c_contiguous
    d = _idx(device_idx)
    h = _idx(host_idx)
    assert d.shape == h.shape
    device_slots = device_layer.size // row_bytes
    host_pages = host.size // (num_layers * page_size * row_bytes)
    rc = lib.oracle_load_layer(num_layers, page_size, row_bytes, device_slots, host_pages, layer,
                               _ptr(device_layer), _ptr(host), _ptr(h), _ptr(d), d.size)
    _check(rc, "oracle_load_layer")


def load_burst(device_layers, host, layer_begin: int, layer_end: int, host_idx, device_idx, *,
               page_size: int, row_bytes: int, lib=None) -> None:
    """Oracle load-back of layers [layer_begin, layer_end) of one tensor, in place."""
    lib = lib or load()
    L = len(device_layers)
    d = _idx(device_idx)
    h = _idx(host_idx)
    assert d.shape == h.shape
    device_slots = device_layers[0].size // row_bytes
    host_pages = host.size // (L * page_size * row_bytes)
    arr = _layers_array(device_layers)
    rc = lib.oracle_load_burst(L, page_size, row_bytes, device_slots, host_pages,
                               layer_begin, layer_end, ctypes.cast(arr, ctypes.c_void_p),
                               _ptr(host), _ptr(h), _ptr(d), d.size)
    _check(rc, "oracle_load_burst")


def pf_backup_all_layers(device_layers, host, device_idx, host_idx, *, row_bytes: int,
                         lib=None) -> None:
    """Oracle all-layer backup into a page_first ([token][layer][row]) host tensor."""
    lib = lib or load()
    L = len(device_layers)
    assert host.dtype == np.uint8 and host.flags.c_contiguous
    d = _idx(device_idx)
    h = _idx(host_idx)
    assert d.shape == h.shape
    device_slots = device_layers[0].size // row_bytes
    host_tokens = host.size // (L * row_bytes)
    arr = _layers_array(device_layers)
    rc = lib.oracle_pf_backup_all_layers(L, row_bytes, device_slots, host_tokens,
                                         ctypes.cast(arr, ctypes.c_void_p), _ptr(host), _ptr(d),
                                         _ptr(h), d.size)
    _check(rc, "oracle_pf_backup_all_layers")


def pf_load_layer(device_layer, host, layer: int, host_idx, device_idx, *, num_layers: int,
                  row_bytes: int, lib=None) -> None:
    """Oracle load-back of one layer from a page_first host tensor."""
    lib = lib or load()
    assert device_layer.dtype == np.uint8 and device_layer.flags.c_contiguous
    d = _idx(device_idx)
    h = _idx(host_idx)
    assert d.shape == h.shape
    device_slots = device_layer.size // row_bytes
    host_tokens = host.size // (num_layers * row_bytes)
    rc = lib.oracle_pf_load_layer(num_layers, row_bytes, device_slots, host_tokens, layer,
                                  _ptr(device_layer), _ptr(host), _ptr(h), _ptr(d), d.size)
    _check(rc, "oracle_pf_load_layer")
