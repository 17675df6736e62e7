"""The seeded input generators and the workload shapes (no GPU).

Both the oracle and the CUDA path are fed from these generators, so their
promises are checked here: destinations are distinct, whole pages are whole
and aligned, exclusions hold, and every workload has the shape the
benchmark reports.
"""
import numpy as np
import pytest

from hierarchical_kv_cache_gb300 import workloads as W


@pytest.mark.parametrize("P", [1, 3, 16, 64])
def test_page_pairs_are_distinct_whole_aligned_pages(P):
    for seed in range(20):
        dev_pages, host_pages, k = 50, 40, 17
        d, h, dp, hp = W.page_pairs(seed, k, dev_pages, host_pages, P)
        assert d.size == h.size == k * P
        assert len(set(d.tolist())) == d.size and len(set(h.tolist())) == h.size
        assert d.min() >= 0 and d.max() < dev_pages * P and h.min() >= 0 and h.max() < host_pages * P
        for side, pages in ((d, dp), (h, hp)):
            blocks = side.reshape(k, P)
            assert (blocks[:, 0] % P == 0).all()
            assert (np.diff(blocks, axis=1) == 1).all()
            assert np.array_equal(blocks[:, 0] // P, pages)
        d2, _, dp2, _ = W.page_pairs(seed + 1, k, dev_pages, host_pages, P, exclude_device_pages=dp)
        assert not set(dp2.tolist()) & set(dp.tolist())


@pytest.mark.parametrize("P", [1, 16, 64])
@pytest.mark.parametrize("fragmented", [False, True])
def test_token_pairs_are_distinct(P, fragmented):
    n, slots = 1000 - 7, 4096
    d, h = W.token_pairs(5, n, slots, slots, P, fragmented=fragmented)
    assert d.size == h.size == n
    assert len(set(d.tolist())) == n and len(set(h.tolist())) == n
    assert 0 <= d.min() and d.max() < slots and 0 <= h.min() and h.max() < slots
    if not fragmented:
        assert np.array_equal(d, np.arange(n)) and np.array_equal(h, np.arange(n))


def test_generators_are_seeded():
    a = W.page_pairs(3, 10, 100, 100, 16)
    b = W.page_pairs(3, 10, 100, 100, 16)
    c = W.page_pairs(4, 10, 100, 100, 16)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0])


def test_workload_shapes():
    llama = W.llama3_8b_mha()
    (s,) = llama.pools
    assert (s.num_layers, s.num_tensors, s.row_bytes, s.page_size) == (32, 2, 2048, 64)
    assert (s.device_slots, s.host_pages, llama.move_pages) == (65536, 1024, 256)
    dsv3 = W.dsv3_mla()
    (s,) = dsv3.pools
    assert (s.num_layers, s.num_tensors, s.row_bytes, s.page_size) == (61, 1, 1152, 64)
    assert (s.host_pages, dsv3.move_pages) == (4096, 512)
    mla = W.mla78_dsa()
    lat, idx = mla.pools
    assert (lat.num_layers, lat.row_bytes, idx.num_layers, idx.row_bytes) == (78, 1152, 78, 132)
    assert idx.page_granular and not lat.page_granular and mla.move_pages == 1024
    assert lat.page_size == idx.page_size == 64
    tiny = W.tiny_mha()
    (s,) = tiny.pools
    assert (s.num_layers, s.num_tensors, s.row_bytes, s.page_size, tiny.move_pages) == (4, 2, 256, 16, 64)
    mamba = W.mamba_state()
    conv, ssm = mamba.pools
    assert conv.page_size == ssm.page_size == 1 and conv.num_layers == ssm.num_layers == 24
    assert conv.row_bytes == 60 * 1024 and ssm.row_bytes == 2 * 1024 * 1024
    assert mamba.move_pages == 32
