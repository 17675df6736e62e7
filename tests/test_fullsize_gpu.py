"""Full-size parity for the DeepSeek-V3, 78-layer two-pool and Mamba state workloads (GPU).

The pools have the benchmark's sizes and the transfers run in the benchmark's
launch configuration: device-located indices, the single-launch burst and the
default grids; the 78-layer workload runs once more with 16 CTAs per launch,
which take the deep tasks.  The oracle then runs on whole-pool images taken before the
transfers, with the workload's own pair lists (no renumbering), and every byte
of both pools is compared, touched and untouched: the host pools after the
backup, the device pools after the load-back burst.  The load-back check feeds
the oracle its own backup result, so no output of the CUDA path becomes an
oracle input.  The host pools start from a position-dependent fill, so a stray
write anywhere would show.  The images need about twice the pools' size in
host memory (26 GB for the 78-layer workload).
"""
import gc

import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import pools as hpools  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_full_size(wl, max_ctas=0):
    shapes = wl.pools
    P = shapes[0].page_size
    L = shapes[0].num_layers
    pools = []
    for i, s in enumerate(shapes):
        p = hpools.allocate_pool(s)
        hpools.fill_device_random_(p, wl.seed + i, s.value_kind)
        hpools.fill_host_pattern_(p, salt=wl.seed + i)
        pools.append(p)
    torch.cuda.synchronize()
    dev_pages = min(s.device_slots for s in shapes) // P
    host_pages = min(s.host_pages for s in shapes)
    d, h, dp, _ = W.page_pairs(wl.seed, wl.move_pages, dev_pages, host_pages, P)
    d2, _, _, _ = W.page_pairs(wl.seed + 1, wl.move_pages, dev_pages, host_pages, P,
                               exclude_device_pages=dp)

    # oracle inputs: whole-pool images, taken before the transfers
    dev_imgs = [G.device_images(p) for p in pools]
    host_imgs = [G.host_images(p) for p in pools]

    words = torch.zeros(4 * L, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    opts = hk.Opts(index_location=hk.HICACHE_INDEX_DEVICE, burst_words=words, device_error=err,
                   max_ctas=max_ctas)
    events = [torch.cuda.Event() for _ in range(L)]
    dt, ht = G.index_tensors(d, h, "device")
    d2t, _ = G.index_tensors(d2, h, "device")
    hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
    hk.hicache_load_burst(pools, 0, L, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert all(e.query() for e in events)

    for i, p in enumerate(pools):
        G.oracle_backup(p, dev_imgs[i], host_imgs[i], d, h)
        G.assert_host_equal(p, host_imgs[i], f"{wl.name}: pool {i} after the backup")
        G.oracle_load(p, dev_imgs[i], host_imgs[i], range(L), h, d2)
        G.assert_device_equal(p, dev_imgs[i], f"{wl.name}: pool {i} after the load-back burst")
        dev_imgs[i] = host_imgs[i] = None
        gc.collect()
    del pools
    gc.collect()
    torch.cuda.empty_cache()


def test_dsv3_mla_full_size():
    _run_full_size(W.dsv3_mla())


def test_mla78_two_pools_full_size():
    _run_full_size(W.mla78_dsa())


def test_mla78_two_pools_full_size_deep_tasks():
    # 16 CTAs per launch: 16-warp CTAs with the deep tasks (4 KiB, 8 chunks in
    # flight per lane)
    _run_full_size(W.mla78_dsa(), max_ctas=16)


def test_mamba_state_pools_full_size():
    _run_full_size(W.mamba_state())
