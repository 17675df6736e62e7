"""The AUTO path rule (hicache_auto_path), host only: no GPU and no CUDA call.

The rule comes from measurements on GB300 with a bf16 GEMM loop occupying
the SMs and without it: zero-copy wins whenever the copy may use enough CTAs
to fill the host link, and the staged path (copy-engine DMA, SMs only for
short gather and scatter kernels) wins when the caller caps the copy's CTAs
below the crossover, provided it may run (staging buffers, host-located
indices, whole host pages) and its DMAs are large (host pages of 1 MiB or
more).  Every condition of the rule is flipped alone here and must flip the
answer back to zero-copy.
"""
import ctypes

import numpy as np
import pytest

import hierarchical_kv_cache_gb300 as hk
from hierarchical_kv_cache_gb300 import _binding as B
from hierarchical_kv_cache_gb300.build import build
from tests.test_abi_cpu import FAKE, c_pool

ZC, ST = hk.HICACHE_PATH_ZERO_COPY, hk.HICACHE_PATH_STAGED
BACKUP, LOAD = hk.HICACHE_OP_BACKUP, hk.HICACHE_OP_LOAD
MiB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def llama_pool(pages=1024, slots=65536):
    # 32 layers x 64 tokens x 2 KiB: 4 MiB host pages per tensor
    return c_pool(L=32, T=2, head_num=8, head_dim=128, dtype_size=2, P=64, slots=slots,
                  pages=pages)


def whole_pages(k, P=64, first_dev=0, first_host=0):
    pages = np.arange(k, dtype=np.int64)
    d = ((pages * 3 + first_dev)[:, None] * P + np.arange(P)).reshape(-1)
    h = ((pages[::-1] + first_host)[:, None] * P + np.arange(P)).reshape(-1)
    return d, h


def opts(max_ctas=4, staging_bytes=256 * MiB, location=hk.HICACHE_INDEX_HOST, path=0):
    o = B.c_opts(path=path, index_location=location, max_ctas=max_ctas, reserved=0)
    if staging_bytes:
        o.staging[0] = FAKE + 0x40000000
        o.staging[1] = FAKE + 0x80000000
        o.staging_bytes = staging_bytes
    return o


def auto(pools, d, h, o, op, layers=32):
    arr = (B.c_pool * len(pools))(*pools)
    d = np.ascontiguousarray(d, dtype=np.int64)
    h = np.ascontiguousarray(h, dtype=np.int64)
    out = ctypes.c_int32(-1)
    st = B.lib().hicache_auto_path(arr, len(pools), d.ctypes.data, h.ctypes.data, 64, d.size,
                                   ctypes.byref(o), op, layers, ctypes.byref(out))
    assert st == hk.HICACHE_OK, B.lib().hicache_last_error().decode()
    return out.value


def test_staged_when_every_condition_holds():
    d, h = whole_pages(256)
    p = [llama_pool()]
    assert auto(p, d, h, opts(), BACKUP) == ST
    assert auto(p, d, h, opts(), LOAD, layers=32) == ST
    assert auto(p, d, h, opts(), LOAD, layers=2) == ST


def test_zero_copy_without_a_cta_cap_or_at_the_crossover():
    d, h = whole_pages(256)
    p = [llama_pool()]
    assert auto(p, d, h, opts(max_ctas=0), BACKUP) == ZC
    assert auto(p, d, h, opts(max_ctas=0), LOAD) == ZC
    b, l = hk.HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP, hk.HICACHE_AUTO_STAGED_BELOW_CTAS_LOAD
    assert auto(p, d, h, opts(max_ctas=b - 1), BACKUP) == ST
    assert auto(p, d, h, opts(max_ctas=b), BACKUP) == ZC
    assert auto(p, d, h, opts(max_ctas=l - 1), LOAD) == ST
    assert auto(p, d, h, opts(max_ctas=l), LOAD) == ZC
    assert auto(p, d, h, opts(max_ctas=152), BACKUP) == ZC


def test_zero_copy_when_the_staged_path_may_not_run():
    d, h = whole_pages(256)
    p = [llama_pool()]
    # no staging buffers
    assert auto(p, d, h, opts(staging_bytes=0), BACKUP) == ZC
    # device-located indices: the DMA spans cannot be planned on the CPU
    assert auto(p, d, h, opts(location=hk.HICACHE_INDEX_DEVICE), BACKUP) == ZC
    # pairs that are not whole host pages: a partial page, then a misaligned page
    assert auto(p, d[:-1], h[:-1], opts(), BACKUP) == ZC
    assert auto(p, d + 1, h + 1, opts(), BACKUP) == ZC
    hh = h.copy()
    hh[5], hh[6] = hh[6], hh[5]  # tokens out of order inside a page
    assert auto(p, d, hh, opts(), BACKUP) == ZC
    # empty list
    assert auto(p, d[:0], h[:0], opts(), BACKUP) == ZC


def test_zero_copy_for_a_single_layer_load():
    d, h = whole_pages(256)
    assert auto([llama_pool()], d, h, opts(), LOAD, layers=1) == ZC


def test_zero_copy_when_host_pages_are_small():
    # 4 layers x 16 tokens x 64 B = 4 KiB host pages: one DMA per page is all fixed cost
    p = [c_pool(L=4, T=1, head_num=1, head_dim=32, dtype_size=2, P=16, slots=4096, pages=512)]
    d, h = whole_pages(64, P=16)
    assert auto(p, d, h, opts(), BACKUP) == ZC
    assert auto(p, d, h, opts(), LOAD, layers=4) == ZC


def test_staging_capacity_is_per_direction():
    d, h = whole_pages(256)
    p = [llama_pool()]
    # 4 MiB holds one layer of a page (2 x 128 KiB) but not a whole page (2 x 4 MiB)
    assert auto(p, d, h, opts(staging_bytes=4 * MiB), BACKUP) == ZC
    assert auto(p, d, h, opts(staging_bytes=4 * MiB), LOAD) == ST
    assert auto(p, d, h, opts(staging_bytes=8 * MiB), BACKUP) == ST


def test_two_pools_latent_beside_a_small_indexer():
    # 78 layers: latent 1152 B rows (5.75 MB pages), indexer 132 B rows page-granular
    lat = c_pool(L=78, T=1, head_num=1, head_dim=576, dtype_size=2, P=64, slots=131072,
                 pages=2048)
    idx = c_pool(L=78, T=1, head_num=1, head_dim=132, dtype_size=1, P=64, slots=131072,
                 pages=2048, page_granular=1)
    d, h = whole_pages(512)
    assert auto([lat, idx], d, h, opts(), BACKUP) == ST
    assert auto([lat, idx], d, h, opts(), LOAD, layers=78) == ST
    # the indexer alone has 659 KB pages: below 1 MiB
    assert auto([idx], d, h, opts(), BACKUP) == ZC


def test_explicit_paths_are_returned_as_given():
    d, h = whole_pages(8)
    p = [llama_pool()]
    assert auto(p, d, h, opts(max_ctas=0, path=ST), BACKUP) == ST
    assert auto(p, d, h, opts(max_ctas=2, path=ZC), BACKUP) == ZC


def test_rejects_bad_arguments():
    d, h = whole_pages(4)
    arr = (B.c_pool * 1)(llama_pool())
    o = opts()
    out = ctypes.c_int32(-1)
    lib = B.lib()
    assert lib.hicache_auto_path(arr, 1, d.ctypes.data, h.ctypes.data, 64, d.size,
                                 ctypes.byref(o), 2, 1, ctypes.byref(out)) == hk.HICACHE_EINVAL
    assert lib.hicache_auto_path(arr, 1, d.ctypes.data, h.ctypes.data, 64, d.size,
                                 ctypes.byref(o), BACKUP, 1, None) == hk.HICACHE_EINVAL
    assert lib.hicache_auto_path(arr, 1, d.ctypes.data, h.ctypes.data, 48, d.size,
                                 ctypes.byref(o), BACKUP, 1, ctypes.byref(out)) == hk.HICACHE_EINVAL
    bad = B.c_opts(path=7, index_location=0)
    assert lib.hicache_auto_path(arr, 1, d.ctypes.data, h.ctypes.data, 64, d.size,
                                 ctypes.byref(bad), BACKUP, 1,
                                 ctypes.byref(out)) == hk.HICACHE_EINVAL


class _Addr:
    """Stands in for a tensor where only its address is read (never dereferenced)."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def test_binding_takes_numpy_host_arrays():
    d, h = whole_pages(256)
    pool = hk.Pool(device_layers=[[_Addr(FAKE + 0x100000 * (t * 32 + l)) for l in range(32)]
                                  for t in range(2)],
                   host_tensors=[_Addr(FAKE + 0x10000000 * (t + 1)) for t in range(2)],
                   num_layers=32, head_num=8, head_dim=128, dtype_size=2, page_size=64,
                   device_slots=65536, host_pages=1024)
    staging = [_Numel(FAKE + 0x40000000), _Numel(FAKE + 0x80000000)]
    o = hk.Opts(max_ctas=4, staging=staging)
    assert hk.hicache_auto_path(pool, d, h, op=BACKUP, opts=o) == ST
    assert hk.hicache_auto_path(pool, d, h, op=LOAD, layers=1, opts=o) == ZC
    assert hk.hicache_auto_path(pool, d, h, op=BACKUP) == ZC
    assert hk.hicache_auto_path(pool, d.astype(np.int32), h.astype(np.int32), op=LOAD,
                                layers=32, opts=o) == ST


class _Numel(_Addr):
    """A 256 MiB staging buffer stand-in."""

    def numel(self):
        return 256 * MiB

    def element_size(self):
        return 1


def test_binding_constants_match_the_header():
    import os
    import re

    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                             "include", "hicache.h")).read()
    for name in ("HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP", "HICACHE_AUTO_STAGED_BELOW_CTAS_LOAD",
                 "HICACHE_OP_BACKUP", "HICACHE_OP_LOAD", "HICACHE_DEVERR_TIMEOUT"):
        m = re.search(r"#define\s+%s\s+(\d+)" % name, text)
        assert m, name
        assert int(m.group(1)) == getattr(hk, name), name
