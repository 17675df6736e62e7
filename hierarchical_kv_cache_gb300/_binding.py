"""Thin ctypes binding of ``libhicache_gb300.so`` (include/hicache.h).

Argument marshalling only: every byte is moved by the library's CUDA kernels or
its copy-engine DMA.  Torch supplies device memory, pinned host memory,
streams and events.  The functions keep the C names and raise ``HiCacheError``
for a non-OK status.  If the library has not been built, every call raises
``RuntimeError``; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhicache_gb300.so")

HICACHE_OK, HICACHE_EINVAL, HICACHE_ERANGE, HICACHE_EDUP, HICACHE_EALIGN, HICACHE_ECUDA, \
    HICACHE_ENOSTAGE = range(7)
STATUS_NAMES = {0: "HICACHE_OK", 1: "HICACHE_EINVAL", 2: "HICACHE_ERANGE", 3: "HICACHE_EDUP",
                4: "HICACHE_EALIGN", 5: "HICACHE_ECUDA", 6: "HICACHE_ENOSTAGE"}
HICACHE_PATH_AUTO, HICACHE_PATH_ZERO_COPY, HICACHE_PATH_STAGED = 0, 1, 2
HICACHE_INDEX_HOST, HICACHE_INDEX_DEVICE = 0, 1
HICACHE_LAYOUT_PAGE_FIRST_DIRECT, HICACHE_LAYOUT_PAGE_FIRST = 0, 1
HICACHE_OP_BACKUP, HICACHE_OP_LOAD = 0, 1
# copy-CTA budgets below which AUTO may take the staged path (include/hicache.h)
HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP, HICACHE_AUTO_STAGED_BELOW_CTAS_LOAD = 5, 5
HICACHE_DEVERR_RANGE, HICACHE_DEVERR_PAGE_ALIGN, HICACHE_DEVERR_TIMEOUT = 1, 2, 4


class c_pool(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_tensors", ctypes.c_int32),
                ("head_num", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype_size", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("page_granular", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("device_slots", ctypes.c_int64), ("host_pages", ctypes.c_int64),
                ("device_layers", ctypes.POINTER(ctypes.c_void_p)),
                ("host_tensors", ctypes.POINTER(ctypes.c_void_p))]


class c_opts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("index_location", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("staging", ctypes.c_void_p * 2), ("staging_bytes", ctypes.c_size_t),
                ("copy_stream", ctypes.c_void_p), ("device_error", ctypes.c_void_p),
                ("burst_words", ctypes.c_void_p), ("burst_words_len", ctypes.c_int64),
                ("index_staging", ctypes.c_void_p), ("index_staging_bytes", ctypes.c_size_t)]


class c_run(ctypes.Structure):
    _fields_ = [("d0", ctypes.c_int64), ("h0", ctypes.c_int64), ("len", ctypes.c_int64)]


_lib = None


def lib():
    """The loaded C library; raises if it was not built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "hierarchical_kv_cache_gb300.build.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        P = ctypes.POINTER(c_pool)
        O = ctypes.POINTER(c_opts)
        L.hicache_backup_all_layers.argtypes = [P, i32, vp, vp, i32, i64, O, vp]
        L.hicache_load_layer.argtypes = [P, i32, i32, vp, vp, i32, i64, O, vp, vp]
        L.hicache_load_burst.argtypes = [P, i32, i32, i32, vp, vp, i32, i64, O, vp,
                                         ctypes.POINTER(vp)]
        L.hicache_plan_runs.argtypes = [vp, vp, i32, i64, i32, ctypes.POINTER(c_run), i64,
                                        ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.hicache_layer_checksum.argtypes = [P, i32, i32, vp, i32, i64, vp, vp]
        L.hicache_check_pairs.argtypes = [P, i32, vp, vp, i32, i64, i32]
        L.hicache_auto_path.argtypes = [P, i32, vp, vp, i32, i64, O, i32, i32,
                                        ctypes.POINTER(i32)]
        L.hicache_auto_path.restype = ctypes.c_int
        L.hicache_backup_all_layers_static_staging.argtypes = [P, i32, vp, vp, i32, i64, O, vp]
        L.hicache_backup_all_layers_static_staging.restype = ctypes.c_int
        for f in ("hicache_backup_all_layers", "hicache_load_layer", "hicache_load_burst",
                  "hicache_plan_runs", "hicache_layer_checksum", "hicache_check_pairs"):
            getattr(L, f).restype = ctypes.c_int
        L.hicache_last_error.restype = ctypes.c_char_p
        L.hicache_last_error.argtypes = []
        L.hicache_abi_version.restype = ctypes.c_int32
        L.hicache_abi_version.argtypes = []
        L.hicache_kernel_launches.restype = ctypes.c_int64
        L.hicache_kernel_launches.argtypes = []
        L.hicache_index_staging_bytes.restype = ctypes.c_size_t
        L.hicache_index_staging_bytes.argtypes = [i64, i32]
        _lib = L
    return _lib


class HiCacheError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


def _check(status: int):
    if status != HICACHE_OK:
        raise HiCacheError(status, lib().hicache_last_error().decode(errors="replace"))


@dataclass
class Pool:
    """One KV pool: device layer buffers [tensor][layer] and pinned host tensors [tensor].

    Any tensor dtype works; the library sees bytes.  device_layers[t][l] must
    hold device_slots * row_bytes bytes and host_tensors[t] host_pages *
    num_layers * page_size * row_bytes bytes, in the host ``layout``
    (HICACHE_LAYOUT_PAGE_FIRST_DIRECT or HICACHE_LAYOUT_PAGE_FIRST).
    """

    device_layers: Sequence[Sequence]
    host_tensors: Sequence
    num_layers: int
    head_num: int
    head_dim: int
    dtype_size: int
    page_size: int
    device_slots: int
    host_pages: int
    page_granular: bool = False
    layout: int = HICACHE_LAYOUT_PAGE_FIRST_DIRECT

    @property
    def num_tensors(self) -> int:
        return len(self.host_tensors)

    @property
    def row_bytes(self) -> int:
        return self.head_num * self.head_dim * self.dtype_size

    def to_c(self):
        """(c_pool, keep): the struct and the pointer arrays it points into.

        The caller holds `keep` until the C call returns.  The last struct built
        is kept on the Pool and reused while every buffer address and shape
        field is unchanged (building the ctypes arrays costs tens of
        microseconds for a pool of many layers); threads may share one Pool.
        """
        T, L = self.num_tensors, self.num_layers
        dev_ptrs = [self.device_layers[t][l].data_ptr() for t in range(T) for l in range(L)]
        host_ptrs = [h.data_ptr() for h in self.host_tensors]
        key = (T, L, self.head_num, self.head_dim, self.dtype_size, self.page_size,
               self.device_slots, self.host_pages, bool(self.page_granular), int(self.layout),
               tuple(dev_ptrs), tuple(host_ptrs))
        cached = self.__dict__.get("_c_cache")
        if cached is not None and cached[0] == key:
            return cached[1], cached[2]
        dev = (ctypes.c_void_p * (T * L))(*dev_ptrs)
        host = (ctypes.c_void_p * T)(*host_ptrs)
        st = c_pool(num_layers=L, num_tensors=T, head_num=self.head_num,
                    head_dim=self.head_dim, dtype_size=self.dtype_size,
                    page_size=self.page_size, page_granular=int(self.page_granular),
                    layout=int(self.layout), device_slots=self.device_slots,
                    host_pages=self.host_pages,
                    device_layers=ctypes.cast(dev, ctypes.POINTER(ctypes.c_void_p)),
                    host_tensors=ctypes.cast(host, ctypes.POINTER(ctypes.c_void_p)))
        self.__dict__["_c_cache"] = (key, st, (dev, host))
        return st, (dev, host)


@dataclass
class Opts:
    """Mirror of hicache_opts; index_location None = inferred from the index tensors."""

    path: int = HICACHE_PATH_AUTO
    index_location: Optional[int] = None
    max_ctas: int = 0
    staging: Optional[Sequence] = None  # two device tensors
    copy_stream: Optional[object] = None  # torch.cuda.Stream
    device_error: Optional[object] = None  # int32/uint32 tensor of one element
    burst_words: Optional[object] = None  # int32 CUDA tensor, >= 4 words per burst layer
    index_staging: Optional[object] = None  # CUDA tensor for copies of host-located indices


def _pools_arg(pools):
    """(array of c_pool, count, keep); keep must outlive the C call."""
    if not isinstance(pools, (list, tuple)):
        pools = [pools]
    built = [p.to_c() for p in pools]
    arr = (c_pool * len(pools))(*[b[0] for b in built])
    return arr, len(pools), [b[1] for b in built]


def _index_bits(t) -> int:
    import torch
    if t.dtype == torch.int32:
        return 32
    if t.dtype == torch.int64:
        return 64
    raise TypeError(f"index tensors must be int32 or int64, got {t.dtype}")


def _opts_arg(opts: Optional[Opts], a, b):
    o = opts or Opts()
    loc = o.index_location
    if loc is None:
        loc = HICACHE_INDEX_DEVICE if a.is_cuda else HICACHE_INDEX_HOST
    c = c_opts(path=o.path, index_location=loc, max_ctas=o.max_ctas, reserved=0)
    if o.staging is not None:
        c.staging[0] = o.staging[0].data_ptr()
        c.staging[1] = o.staging[1].data_ptr()
        c.staging_bytes = min(o.staging[0].numel() * o.staging[0].element_size(),
                              o.staging[1].numel() * o.staging[1].element_size())
    if o.copy_stream is not None:
        c.copy_stream = o.copy_stream.cuda_stream
    if o.device_error is not None:
        c.device_error = o.device_error.data_ptr()
    if o.burst_words is not None:
        c.burst_words = o.burst_words.data_ptr()
        c.burst_words_len = o.burst_words.numel() * o.burst_words.element_size() // 4
    if o.index_staging is not None:
        c.index_staging = o.index_staging.data_ptr()
        c.index_staging_bytes = o.index_staging.numel() * o.index_staging.element_size()
    return c


def _stream_arg(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _event_handle(ev, stream_handle) -> int:
    """Raw cudaEvent_t of a torch event, creating it on first use."""
    if ev is None:
        return 0
    h = ev.cuda_event
    if h == 0:  # torch creates the CUDA event lazily, on its first record
        ev.record()
        h = ev.cuda_event
    return h


def _indices(a, b):
    if a.numel() != b.numel():
        raise ValueError("index tensors differ in length")
    if a.device != b.device or a.dtype != b.dtype:
        raise ValueError("index tensors must share device and dtype")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("index tensors must be contiguous")
    return _index_bits(a), a.numel()


def hicache_backup_all_layers(pools, device_indices, host_indices, *, opts: Optional[Opts] = None,
                              stream=None) -> None:
    """All-layer D2H backup of pairs device_indices[i] -> host_indices[i] (see hicache.h)."""
    arr, npools, keep = _pools_arg(pools)
    bits, n = _indices(device_indices, host_indices)
    o = _opts_arg(opts, device_indices, host_indices)
    _check(lib().hicache_backup_all_layers(arr, npools, device_indices.data_ptr(),
                                           host_indices.data_ptr(), bits, n, ctypes.byref(o),
                                           _stream_arg(stream)))
    del keep  # the pointer arrays lived until the call returned


def hicache_backup_all_layers_static_staging(pools, device_indices, host_indices, *,
                                             opts: Optional[Opts] = None, stream=None) -> None:
    """All-layer backup through the staged path using the library's own static staging.

    For callers that cannot allocate device memory when they transfer (for
    example an engine that gave all free HBM to its KV pool at start-up): no
    staging buffer is passed and nothing is allocated.  Indices must be pinned
    host tensors covering whole host pages; one host page of all layers must fit
    in 16 MiB.  Calls that overlap on the GPU share the static array and race.
    """
    arr, npools, keep = _pools_arg(pools)
    bits, n = _indices(device_indices, host_indices)
    o = _opts_arg(opts, device_indices, host_indices)
    _check(lib().hicache_backup_all_layers_static_staging(
        arr, npools, device_indices.data_ptr(), host_indices.data_ptr(), bits, n,
        ctypes.byref(o), _stream_arg(stream)))
    del keep  # the pointer arrays lived until the call returned


def hicache_load_layer(pools, layer: int, host_indices, device_indices, *,
                       opts: Optional[Opts] = None, stream=None, layer_done=None) -> None:
    """H2D load-back of one layer; records ``layer_done`` (a torch.cuda.Event) after it."""
    arr, npools, keep = _pools_arg(pools)
    bits, n = _indices(device_indices, host_indices)
    o = _opts_arg(opts, device_indices, host_indices)
    s = _stream_arg(stream)
    _check(lib().hicache_load_layer(arr, npools, layer, host_indices.data_ptr(),
                                    device_indices.data_ptr(), bits, n, ctypes.byref(o), s,
                                    _event_handle(layer_done, s)))
    del keep  # the pointer arrays lived until the call returned


def hicache_load_burst(pools, layer_begin: int, layer_end: int, host_indices, device_indices, *,
                       opts: Optional[Opts] = None, stream=None, layer_done=None) -> None:
    """H2D load-back of layers [layer_begin, layer_end), one event per layer (list or None)."""
    arr, npools, keep = _pools_arg(pools)
    bits, n = _indices(device_indices, host_indices)
    o = _opts_arg(opts, device_indices, host_indices)
    s = _stream_arg(stream)
    count = max(0, layer_end - layer_begin)
    evs = None
    if layer_done is not None:
        if len(layer_done) != count:
            raise ValueError("layer_done must hold one event per layer")
        evs = (ctypes.c_void_p * max(1, count))(*[_event_handle(e, s) for e in layer_done])
    _check(lib().hicache_load_burst(arr, npools, layer_begin, layer_end, host_indices.data_ptr(),
                                    device_indices.data_ptr(), bits, n, ctypes.byref(o), s, evs))
    del keep  # the pointer arrays lived until the call returned


def hicache_plan_runs(device_indices, host_indices, page_size: int):
    """Maximal runs (d0, h0, len) of host-memory index arrays and the whole-page run count."""
    d = np.ascontiguousarray(device_indices)
    h = np.ascontiguousarray(host_indices)
    if d.dtype != h.dtype or d.dtype not in (np.int32, np.int64) or d.shape != h.shape:
        raise TypeError("index arrays must be equal-length int32 or int64")
    bits = 32 if d.dtype == np.int32 else 64
    count = ctypes.c_int64(0)
    full = ctypes.c_int64(0)
    _check(lib().hicache_plan_runs(d.ctypes.data, h.ctypes.data, bits, d.size, page_size, None, 0,
                                   ctypes.byref(count), None))
    runs = (c_run * max(1, count.value))()
    _check(lib().hicache_plan_runs(d.ctypes.data, h.ctypes.data, bits, d.size, page_size, runs,
                                   count.value, ctypes.byref(count), ctypes.byref(full)))
    out = np.array([(r.d0, r.h0, r.len) for r in runs[:count.value]], dtype=np.int64)
    return out.reshape(-1, 3), full.value


def hicache_check_pairs(pools, device_indices, host_indices, *, dest_is_device: bool) -> None:
    """Host-only validation of a pair list in host memory, as a call with host-located
    indices does it; raises HiCacheError with that call's status."""
    arr, n, keep = _pools_arg(pools)
    d = np.ascontiguousarray(device_indices)
    h = np.ascontiguousarray(host_indices)
    if d.dtype != h.dtype or d.dtype not in (np.int32, np.int64) or d.shape != h.shape:
        raise TypeError("index arrays must be equal-length int32 or int64")
    bits = 32 if d.dtype == np.int32 else 64
    _check(lib().hicache_check_pairs(arr, n, d.ctypes.data, h.ctypes.data, bits, d.size,
                                     int(bool(dest_is_device))))
    del keep  # the pointer arrays lived until the call returned


def hicache_auto_path(pools, device_indices, host_indices, *, op: int, layers: int = 1,
                      opts: Optional[Opts] = None) -> int:
    """Path a call with opts.path AUTO takes (host only): HICACHE_PATH_ZERO_COPY or _STAGED.

    Index arrays are numpy arrays (host memory; opts.index_location defaults to
    HICACHE_INDEX_HOST) or torch tensors (location inferred as for the calls).
    """
    arr, npools, keep = _pools_arg(pools)
    if isinstance(device_indices, np.ndarray) or isinstance(host_indices, np.ndarray):
        d = np.ascontiguousarray(device_indices)
        h = np.ascontiguousarray(host_indices)
        if d.dtype != h.dtype or d.dtype not in (np.int32, np.int64) or d.shape != h.shape:
            raise TypeError("index arrays must be equal-length int32 or int64")
        bits, n, dp, hp = 32 if d.dtype == np.int32 else 64, d.size, d.ctypes.data, h.ctypes.data
        o = opts or Opts()
        if o.index_location is None:
            from dataclasses import replace
            o = replace(o, index_location=HICACHE_INDEX_HOST)
        co = _opts_arg(o, None, None)
    else:
        bits, n = _indices(device_indices, host_indices)
        dp, hp = device_indices.data_ptr(), host_indices.data_ptr()
        co = _opts_arg(opts, device_indices, host_indices)
    out = ctypes.c_int32(-1)
    _check(lib().hicache_auto_path(arr, npools, dp, hp, bits, n, ctypes.byref(co), int(op),
                                   int(layers), ctypes.byref(out)))
    del keep  # the pointer arrays lived until the call returned
    return out.value


def hicache_layer_checksum(pool: Pool, tensor: int, layer: int, device_indices, out_sum, *,
                           stream=None) -> None:
    """Adds the 32-bit words of the indexed rows into ``out_sum`` (a zeroed int64 CUDA tensor)."""
    arr, _, keep = _pools_arg(pool)
    bits = _index_bits(device_indices)
    _check(lib().hicache_layer_checksum(arr, tensor, layer, device_indices.data_ptr(), bits,
                                        device_indices.numel(), out_sum.data_ptr(),
                                        _stream_arg(stream)))
    del keep  # the pointer arrays lived until the call returned


def abi_version() -> int:
    return lib().hicache_abi_version()


def index_staging_bytes(n: int, index_bits: int = 64) -> int:
    """Bytes of Opts.index_staging a call with n pairs needs."""
    return lib().hicache_index_staging_bytes(n, index_bits)


def kernel_launches() -> int:
    """Kernels the library has launched in this process."""
    return lib().hicache_kernel_launches()
