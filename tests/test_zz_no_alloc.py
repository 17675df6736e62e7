"""The allocation-free backup entry point (GPU).

hicache_backup_all_layers_static_staging serves callers that cannot allocate
device memory when they transfer: for example a serving engine that handed
all free HBM to its KV pool at start-up, where any later cudaMalloc would fail,
or a thin C caller that has no device allocator of its own.  It stages through
an array the library defines statically instead of caller buffers.

Checked here:
  - on two calls in a row (the second reuses the array the first one left
    behind), the host pool equals, byte for byte, both the CPU oracle's backup
    of the same pairs and what hicache_backup_all_layers writes;
  - page counts whose staged part (all but the last quarter of the pages, which
    move zero-copy) lies just below, on and just past the 16 MiB half of the
    array, and a list of three chunks, so that one call refills a half it used
    before;
  - in a fresh process, once a call with no pairs has done the set-up, later
    calls take no device memory at all.

This file is collected last on purpose, and it needs nothing from the other
test files, so it passes alone in a fresh process too.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import pools as hpools  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


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


def _oracle_backup(pool, dev_imgs, host_imgs, d, h):
    import oracle

    for t in range(pool.num_tensors):
        oracle.backup_all_layers(dev_imgs[t], host_imgs[t], d, h, page_size=pool.page_size,
                                 row_bytes=pool.row_bytes)


def _mha_shape():
    # 2 tensors x 8 layers x 64 tokens x 512 B = 512 KiB per host page: exactly 32 pages
    # fill one 16 MiB half of the static array
    return [W.PoolShape("mha", num_layers=8, num_tensors=2, head_num=4, head_dim=128,
                        dtype_size=1, page_size=64, device_slots=64 * 128, host_pages=100)]


def _mla_dsa_shapes():
    lat = W.PoolShape("mla", num_layers=6, num_tensors=1, head_num=1, head_dim=576,
                      dtype_size=2, page_size=64, device_slots=64 * 64, host_pages=60)
    idx = W.PoolShape("dsa", num_layers=6, num_tensors=1, head_num=1, head_dim=132,
                      dtype_size=1, page_size=64, device_slots=64 * 64, host_pages=60,
                      page_granular=True, value_kind="uint8_uniform")
    return [lat, idx]


# (shapes, pages per call).  The staged backup moves the last ceil(pages / 4) pages
# zero-copy, so 42 / 43 / 44 pages put 31 / 32 / 33 pages through the array: just
# below, on and one past a half.  87 pages put 65 through it, three chunks (32 + 32
# + 1), so the third refills the first half within one call.  The two-pool case has
# 481.5 KiB pages, 34 per half; 50 pages put 37 through it, over both halves.
CASES = {"mha42": (_mha_shape, 42), "mha43": (_mha_shape, 43), "mha44": (_mha_shape, 44),
         "mha87": (_mha_shape, 87), "mla_dsa50": (_mla_dsa_shapes, 50)}


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_staging_matches_oracle_and_backup_twice(case):
    make_shapes, moves = CASES[case]
    shapes = make_shapes()
    P = shapes[0].page_size
    ours, ref = _twin_pools(shapes, seed=31)
    dev_imgs = [[[b.cpu().numpy().copy() for b in per_t] for per_t in p.device_layers]
                for p in ours]
    host_imgs = [[h.numpy().copy() for h in p.host_tensors] for p in ours]
    dev_pages = min(s.device_slots for s in shapes) // P
    host_pages = min(s.host_pages for s in shapes)
    stream = torch.cuda.current_stream()
    for call in range(2):
        d, h, _, _ = W.page_pairs(40 + call, moves, dev_pages, host_pages, P)
        dt, ht = _pinned(d), _pinned(h)
        hk.hicache_backup_all_layers_static_staging(ours, dt, ht, stream=stream)
        hk.hicache_backup_all_layers(ref, dt, ht, stream=stream)
        torch.cuda.synchronize()
        for p, pool in enumerate(ours):
            _oracle_backup(pool, dev_imgs[p], host_imgs[p], d, h)
            for t in range(pool.num_tensors):
                got = pool.host_tensors[t].numpy()
                bad = np.flatnonzero(got != host_imgs[p][t])
                assert bad.size == 0, (f"{case} call {call}: pool {p} tensor {t} differs from the "
                                       f"oracle at {bad.size} bytes, first {bad[:8]}")
                assert torch.equal(pool.host_tensors[t], ref[p].host_tensors[t]), \
                    f"{case} call {call}: pool {p} tensor {t} differs from the staged backup"


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


def test_static_staging_takes_no_device_memory_after_warm_up():
    """In a fresh process: after one call with no pairs, calls take no device memory.

    A fresh process is the case that matters: nothing has loaded the library's
    modules yet, so any lazily placed code or data would show up here as a drop
    in the device's free memory between the warm-up and the later calls.
    """
    r = subprocess.run([sys.executable, os.path.join(HERE, "no_alloc_child.py")],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
    rec = json.loads(line)
    assert rec["moved_ok"], rec
    assert rec["free_after_calls"] == rec["free_after_warm_up"], rec
    assert rec["torch_reserved_after_calls"] == rec["torch_reserved_after_warm_up"], rec
