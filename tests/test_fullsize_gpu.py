"""Full-size parity for the DeepSeek-V3, 78-layer two-pool and Mamba state workloads (GPU).

The pools have the benchmark's sizes and the transfers run in the benchmark's
launch configuration: device-located indices, the single-launch burst and the
default grids.  The oracle computes every touched output one by one on compact
images:
- the device rows the backup reads are gathered into a compact device image;
- the host pages it writes are copied into a compact host image;
- the oracle runs on those images with renumbered indices.
The load-back check then feeds the oracle its own backup result, so no output
of the CUDA path becomes an oracle input.  A seeded sample of untouched host
pages and device rows must keep its bytes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
import oracle  # noqa: E402
from hierarchical_kv_cache_gb300 import pools as hpools  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rows(buf, R):
    return buf.view(-1, R)


def _host_pages(pool, t):
    """Host tensor t as [page][page bytes] (both layouts keep a page contiguous)."""
    return pool.host_tensors[t].view(pool.host_pages, -1)


def _oracle_backup_compact(pool, t, dev_rows, hp, P):
    """Expected bytes of host pages hp (all layers) after the backup, via the oracle.

    dev_rows[l] holds the n source rows of layer l in pair order; the compact
    host image holds exactly the pages hp, renumbered 0..k-1 in that order.
    """
    k = hp.size
    n = k * P
    R = pool.row_bytes
    compact_host = _host_pages(pool, t)[torch.as_tensor(hp)].numpy().reshape(-1).copy()
    d_c = np.arange(n, dtype=np.int64)
    h_c = np.arange(n, dtype=np.int64)  # compact page j holds host page hp[j]
    layers = [np.ascontiguousarray(x.reshape(-1)) for x in dev_rows]
    if pool.layout == 1:
        oracle.pf_backup_all_layers(layers, compact_host, d_c, h_c, row_bytes=R)
    else:
        oracle.backup_all_layers(layers, compact_host, d_c, h_c, page_size=P, row_bytes=R)
    return compact_host


def _oracle_load_compact(pool, compact_host, l, k, P):
    """Expected n loaded rows of layer l (in pair order) from a compact host image."""
    n = k * P
    R = pool.row_bytes
    out = np.zeros(n * R, dtype=np.uint8)
    idx = np.arange(n, dtype=np.int64)
    if pool.layout == 1:
        oracle.pf_load_layer(out, compact_host, l, idx, idx, num_layers=pool.num_layers,
                             row_bytes=R)
    else:
        oracle.load_layer(out, compact_host, l, idx, idx, num_layers=pool.num_layers,
                          page_size=P, row_bytes=R)
    return out.reshape(n, R)


def _run_full_size(wl, sample_pages=48, sample_rows=512):
    shapes = wl.pools
    P = shapes[0].page_size
    pools = []
    for i, s in enumerate(shapes):
        p = hpools.allocate_pool(s)
        hpools.fill_device_random_(p, wl.seed + i, s.value_kind)
        pools.append(p)
    torch.cuda.synchronize()
    dev_pages = min(s.device_slots for s in shapes) // P
    host_pages = min(s.host_pages for s in shapes)
    d, h, dp, hp = W.page_pairs(wl.seed, wl.move_pages, dev_pages, host_pages, P)
    d2, _, dp2, _ = W.page_pairs(wl.seed + 1, wl.move_pages, dev_pages, host_pages, P,
                                 exclude_device_pages=dp)
    n = d.size
    L = shapes[0].num_layers
    g = np.random.default_rng(wl.seed + 2)
    untouched_hp = g.choice(np.setdiff1d(np.arange(host_pages), hp), size=sample_pages,
                            replace=False)
    untouched_rows = g.choice(np.setdiff1d(np.arange(dev_pages * P), d2), size=sample_rows,
                              replace=False)
    dt = torch.as_tensor(d).cuda()
    d_t = torch.as_tensor(d)
    d2_t = torch.as_tensor(d2)

    # oracle inputs, taken from the pools before the transfers
    expect_host, before_host, before_dev = [], [], []
    for p in pools:
        R = p.row_bytes
        per_tensor = []
        for t in range(p.num_tensors):
            rows = [_rows(p.device_layers[t][l], R)[dt].cpu().numpy() for l in range(L)]
            per_tensor.append(_oracle_backup_compact(p, t, rows, hp, P))
        expect_host.append(per_tensor)
        before_host.append([_host_pages(p, t)[torch.as_tensor(untouched_hp)].clone()
                            for t in range(p.num_tensors)])
        before_dev.append([[_rows(p.device_layers[t][l], R)[torch.as_tensor(untouched_rows).cuda()]
                            .cpu() for l in range(L)] for t in range(p.num_tensors)])

    words = torch.zeros(4 * L, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    opts = hk.Opts(index_location=hk.HICACHE_INDEX_DEVICE, burst_words=words, device_error=err)
    events = [torch.cuda.Event() for _ in range(L)]
    ht = torch.as_tensor(h).cuda()
    d2t = torch.as_tensor(d2).cuda()
    hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
    hk.hicache_load_burst(pools, 0, L, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert all(e.query() for e in events)

    for pi, p in enumerate(pools):
        R = p.row_bytes
        for t in range(p.num_tensors):
            got = _host_pages(p, t)[torch.as_tensor(hp)].numpy().reshape(-1)
            assert np.array_equal(got, expect_host[pi][t]), f"pool {pi} tensor {t}: backup pages"
            assert torch.equal(_host_pages(p, t)[torch.as_tensor(untouched_hp)],
                               before_host[pi][t]), f"pool {pi} tensor {t}: untouched pages"
            for l in range(L):
                want = _oracle_load_compact(p, expect_host[pi][t], l, hp.size, P)
                got_rows = _rows(p.device_layers[t][l], R)[d2t].cpu().numpy()
                assert np.array_equal(got_rows, want), f"pool {pi} tensor {t} layer {l}: load"
                assert torch.equal(
                    _rows(p.device_layers[t][l], R)[torch.as_tensor(untouched_rows).cuda()].cpu(),
                    before_dev[pi][t][l]), f"pool {pi} tensor {t} layer {l}: untouched rows"
    del pools
    torch.cuda.empty_cache()
    _ = (d_t, d2_t, dp2)


def test_dsv3_mla_full_size():
    _run_full_size(W.dsv3_mla())


def test_mla78_two_pools_full_size():
    _run_full_size(W.mla78_dsa())


def test_mamba_state_pools_full_size():
    _run_full_size(W.mamba_state(), sample_pages=16, sample_rows=16)
