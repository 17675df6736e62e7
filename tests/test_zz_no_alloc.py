"""The allocation-free backup entry point against the existing one (GPU).

hicache_backup_all_layers_static_staging serves callers that cannot allocate
device memory when they transfer: it stages through an array the library
defines statically instead of caller buffers.  Its output must equal, byte
for byte, what hicache_backup_all_layers writes for the same pools and pairs,
on two calls in a row (the second call reuses the array the first one left
behind).  This file is collected last on purpose, and it needs nothing from
the other test files, so it passes alone in a fresh process too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import pools as hpools  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _twin_pools(shapes, seed):
    """Two pools per shape with identical device bytes and identical host fill."""
    a = [hpools.allocate_pool(s) for s in shapes]
    b = [hpools.allocate_pool(s) for s in shapes]
    for i, (pa, pb, s) in enumerate(zip(a, b, shapes)):
        hpools.fill_device_random_(pa, seed + i, s.value_kind)
        hpools.fill_host_pattern_(pa, salt=seed + i)
        for t in range(pa.num_tensors):
            pb.host_tensors[t].copy_(pa.host_tensors[t])
            for l in range(pa.num_layers):
                pb.device_layers[t][l].copy_(pa.device_layers[t][l])
    torch.cuda.synchronize()
    return a, b


def _pinned(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int64)).pin_memory()


def _assert_same_host(a, b, what):
    for pa, pb in zip(a, b):
        for t in range(pa.num_tensors):
            assert torch.equal(pa.host_tensors[t], pb.host_tensors[t]), f"{what}: tensor {t}"


@pytest.mark.parametrize("case", ["mha", "mla_dsa"])
def test_static_staging_matches_backup_twice(case):
    if case == "mha":
        # 2 tensors x 8 layers x 64 tokens x 512 B = 512 KiB per host page: 32 pages per
        # 16 MiB half, so 40 pages use both halves
        shapes = [W.PoolShape("mha", num_layers=8, num_tensors=2, head_num=4, head_dim=128,
                              dtype_size=1, page_size=64, device_slots=64 * 96, host_pages=80)]
        moves = 40
    else:
        lat = W.PoolShape("mla", num_layers=6, num_tensors=1, head_num=1, head_dim=576,
                          dtype_size=2, page_size=64, device_slots=64 * 64, host_pages=60)
        idx = W.PoolShape("dsa", num_layers=6, num_tensors=1, head_num=1, head_dim=132,
                          dtype_size=1, page_size=64, device_slots=64 * 64, host_pages=60,
                          page_granular=True, value_kind="uint8_uniform")
        shapes = [lat, idx]
        moves = 50  # 481.5 KiB per host page: 34 pages per half, so both halves are used
    P = shapes[0].page_size
    ours, ref = _twin_pools(shapes, seed=31)
    dev_pages = min(s.device_slots for s in shapes) // P
    host_pages = min(s.host_pages for s in shapes)
    stream = torch.cuda.current_stream()
    for call in range(2):
        d, h, _, _ = W.page_pairs(40 + call, moves, dev_pages, host_pages, P)
        dt, ht = _pinned(d), _pinned(h)
        hk.hicache_backup_all_layers_static_staging(ours, dt, ht, stream=stream)
        hk.hicache_backup_all_layers(ref, dt, ht, stream=stream)
        torch.cuda.synchronize()
        _assert_same_host(ours, ref, f"{case} call {call}")


def test_static_staging_rejects_pages_above_its_half():
    # 2 tensors x 64 layers x 64 tokens x 4 KiB = 32 MiB per host page, above 16 MiB
    s = W.PoolShape("big", num_layers=64, num_tensors=2, head_num=16, head_dim=128,
                    dtype_size=2, page_size=64, device_slots=128, host_pages=2)
    pool = hpools.allocate_pool(s)
    d, h, _, _ = W.page_pairs(50, 1, 2, 2, 64)
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_backup_all_layers_static_staging(pool, _pinned(d), _pinned(h))
    assert ei.value.status == hk.HICACHE_ENOSTAGE
    assert "static staging array" in ei.value.message
