"""Seeded random parity cases through the CUDA path (GPU).

Each case draws, from its seed, a pool shape, an index type and location, a
path and a layer range.  It runs an all-layer backup and a load-back burst
through the C ABI and compares every byte of every pool with the CPU oracle
applied to copies of the pools taken before each call.  The draws reach
combinations the hand-written cases do not:
- row sizes that take 16-byte or 4-byte chunks, and rows longer than a task;
- page sizes 1 to 64, both host layouts, page-granular pools;
- one or two pools in a call, whole or partial last pages, repeated backup
  sources;
- sub-ranges of layers, including an empty one;
- every path that accepts the draw: one launch per layer, the single-launch
  burst, and the staged path with staging from one page up.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as G  # noqa: E402

pytestmark = pytest.mark.gpu

CASES = 160
# (head_num, head_dim, dtype_size): rows of 4, 12, 16, 36, 64, 132, 256, 1152, 2048 and
# 8196 bytes; 4, 12, 36, 132 and 8196 are not multiples of 16 (4-byte chunks)
ROWS = [(1, 2, 2), (1, 6, 2), (1, 8, 2), (1, 18, 2), (2, 16, 2), (1, 132, 1), (2, 64, 2),
        (1, 576, 2), (8, 128, 2), (1, 4098, 2)]
POOL_BYTES = 24 << 20  # cap on device bytes per pool (all layers and tensors)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _draw(seed):
    g = np.random.default_rng(7000 + seed)
    L = int(g.integers(1, 10))
    P = int(g.choice([1, 2, 3, 8, 16, 64]))
    npools = int(g.choice([1, 1, 2]))
    path = str(g.choice(["per_layer", "single_launch", "staged"]))
    where = str(g.choice(["device", "host", "host_staged_idx"]))
    if path == "staged" and where == "device":
        where = "host"  # the staged path plans its copies on the CPU
    shapes = []
    for i in range(npools):
        hn, hd, ds = ROWS[int(g.integers(0, len(ROWS)))]
        T = int(g.integers(1, 3))
        layout = str(g.choice(["page_first_direct", "page_first"]))
        granular = bool(P > 1 and g.random() < 0.25)
        shapes.append(dict(T=T, head_num=hn, head_dim=hd, dtype_size=ds, layout=layout,
                           page_granular=granular, name=f"p{i}"))
    whole_pages = path == "staged" or any(s["page_granular"] for s in shapes) or g.random() < 0.3
    # pages moved, bounded so that every pool stays within POOL_BYTES
    max_row = max(s["head_num"] * s["head_dim"] * s["dtype_size"] * s["T"] for s in shapes)
    max_slots = max(4 * P, POOL_BYTES // (max_row * L))
    k = int(g.integers(1, max(2, min(40, max_slots // (3 * P)))))
    dev_pages = 2 * k + int(g.integers(0, 8))
    host_pages = k + int(g.integers(0, 12))
    idx_dtype = torch.int32 if g.random() < 0.5 else torch.int64
    l0 = int(g.integers(0, L))
    l1 = int(g.integers(l0 + 1, L + 1)) if g.random() > 0.05 else l0  # now and then empty
    return g, dict(L=L, P=P, shapes=shapes, path=path, where=where, whole_pages=whole_pages, k=k,
                   dev_pages=dev_pages, host_pages=host_pages, idx_dtype=idx_dtype, l0=l0, l1=l1)


@pytest.mark.parametrize("seed", range(CASES))
def test_random_case(seed):
    g, c = _draw(seed)
    L, P, k = c["L"], c["P"], c["k"]
    slots = c["dev_pages"] * P
    pools = []
    for i, s in enumerate(c["shapes"]):
        shape = G.shape(s["name"], L=L, T=s["T"], head_num=s["head_num"], head_dim=s["head_dim"],
                        dtype_size=s["dtype_size"], P=P, slots=slots, pages=c["host_pages"],
                        page_granular=s["page_granular"], layout=s["layout"],
                        value_kind="uint8_uniform" if s["page_granular"] else "bf16_normal")
        pools.append(G.make_pool(shape, seed=100 * seed + i))

    # backup pairs: whole pages, or tokens of random pages with a partial last
    # page and some repeated device sources
    if c["whole_pages"]:
        d, h, dp, _ = W.page_pairs(seed, k, c["dev_pages"], c["host_pages"], P)
    else:
        n = k * P - int(g.integers(0, P))
        d, h = W.token_pairs(seed, n, slots, c["host_pages"] * P, P, fragmented=True)
        d = d.copy()
        if n > 2:
            d[g.integers(0, n, size=n // 5)] = d[0]
        dp = np.unique(d // P)
    n = d.size
    # load-back destinations: other device pages (whole pages for page-granular
    # pools), or distinct random device slots
    if c["whole_pages"]:
        d2, _, _, _ = W.page_pairs(seed + 1, k, c["dev_pages"], c["host_pages"], P,
                                   exclude_device_pages=dp)
        d2 = d2[:n]
    else:
        d2 = g.choice(slots, size=n, replace=False).astype(np.int64)

    where = "host" if c["where"] == "host_staged_idx" else c["where"]
    dt, ht = G.index_tensors(d, h, where, c["idx_dtype"])
    d2t, _ = G.index_tensors(d2, h, where, c["idx_dtype"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(device_error=err)
    if c["where"] == "host_staged_idx":
        bits = 32 if c["idx_dtype"] == torch.int32 else 64
        kw["index_staging"] = torch.empty(hk.index_staging_bytes(n, bits), dtype=torch.uint8,
                                          device="cuda")
    if c["path"] == "staged":
        per_page = sum(p.num_tensors * L * P * p.row_bytes for p in pools)
        cap = int(g.integers(1, k + 3))
        kw["staging"] = [torch.empty(cap * per_page + int(g.integers(0, 64)) * 16,
                                     dtype=torch.uint8, device="cuda") for _ in range(2)]
        path = hk.HICACHE_PATH_STAGED
    else:
        path = hk.HICACHE_PATH_ZERO_COPY
        if c["path"] == "single_launch":
            kw["burst_words"] = torch.full((4 * L,), 7, dtype=torch.int32, device="cuda")
    loc = hk.HICACHE_INDEX_DEVICE if where == "device" else hk.HICACHE_INDEX_HOST
    opts = hk.Opts(path=path, index_location=loc, **kw)
    what = f"seed {seed}: {c}"

    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]
    host_before = [G.host_images(p) for p in pools]
    hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
    torch.cuda.synchronize()
    for p, (dev0, host0) in zip(pools, imgs):
        G.oracle_backup(p, dev0, host0, d, h)
        G.assert_host_equal(p, host0, "backup " + what)
    # the case moved something: random device rows replaced the host fill pattern
    assert any(not np.array_equal(a, b) for (_, host0), hb in zip(imgs, host_before)
               for a, b in zip(host0, hb)), what

    dev1 = [G.device_images(p) for p in pools]
    dev_before = [[[x.copy() for x in per_t] for per_t in dv] for dv in dev1]
    events = [torch.cuda.Event() for _ in range(c["l1"] - c["l0"])]
    hk.hicache_load_burst(pools, c["l0"], c["l1"], ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, what
    for p, dv, (_, host0) in zip(pools, dev1, imgs):
        G.oracle_load(p, dv, host0, range(c["l0"], c["l1"]), h, d2)
        G.assert_device_equal(p, dv, "burst " + what)
    if c["l1"] > c["l0"]:
        assert any(not np.array_equal(a, b) for dv, db in zip(dev1, dev_before)
                   for per_a, per_b in zip(dv, db) for a, b in zip(per_a, per_b)), what


REJECT_CASES = 48
FAULTS = ["dup_destination", "out_of_range", "negative", "partial_page", "layer_range"]


@pytest.mark.parametrize("seed", range(REJECT_CASES))
def test_random_fault(seed):
    """One planted fault in a random case.

    Host-located indices: the call fails with the fault's status, records every
    layer event (checked behind a sleep kernel), and moves no byte.
    Device-located indices (out-of-range and negative entries only): the
    kernels skip the bad pairs, flag them in the error word, and move every
    other pair.
    """
    g, c = _draw(10_000 + seed)
    L, P, k = c["L"], c["P"], c["k"]
    fault = FAULTS[seed % len(FAULTS)]
    on_device = c["where"] == "device" and fault in ("out_of_range", "negative")
    where = "device" if on_device else "host"
    path = c["path"]
    if fault == "partial_page":
        if P == 1:
            fault = "dup_destination"
        elif path != "staged" and not any(s["page_granular"] for s in c["shapes"]):
            path = "staged"  # whole host pages are required there
    slots = c["dev_pages"] * P
    pools = [G.make_pool(G.shape(s["name"], L=L, T=s["T"], head_num=s["head_num"],
                                 head_dim=s["head_dim"], dtype_size=s["dtype_size"], P=P,
                                 slots=slots, pages=c["host_pages"],
                                 page_granular=s["page_granular"], layout=s["layout"],
                                 value_kind="uint8_uniform" if s["page_granular"]
                                 else "bf16_normal"), seed=200 * seed + i)
             for i, s in enumerate(c["shapes"])]
    d, h, dp, _ = W.page_pairs(seed, k, c["dev_pages"], c["host_pages"], P)
    d2, _, _, _ = W.page_pairs(seed + 1, k, c["dev_pages"], c["host_pages"], P,
                               exclude_device_pages=dp)
    d, h, d2 = d.copy(), h.copy(), d2.copy()
    n = d.size
    # on the device the bad pair starts a page: a page-granular pool in the
    # direct layout reads only the first pair of each page
    i = int(g.integers(0, k)) * P if on_device else int(g.integers(0, n))
    l0, l1 = 0, L
    want = hk.HICACHE_EINVAL
    if fault == "dup_destination":
        if n < 2:
            d, h, d2 = np.r_[d, d], np.r_[h, h], np.r_[d2, d2]  # the same pair twice
        else:
            j = (i + 1 + int(g.integers(0, n - 1))) % n
            h[j], d2[j] = h[i], d2[i]
        want = hk.HICACHE_EDUP
    elif fault == "out_of_range":
        h[i] = c["host_pages"] * P + int(g.integers(0, 1000))
        d2[i] = slots + int(g.integers(0, 1000))
        want = hk.HICACHE_ERANGE
    elif fault == "negative":
        h[i] = -1 - int(g.integers(0, 1000))
        d2[i] = -1
        want = hk.HICACHE_ERANGE
    elif fault == "partial_page":
        d, h, d2 = d[:-1], h[:-1], d2[:-1]
    else:
        l0, l1 = int(g.integers(0, L)), L + 1 + int(g.integers(0, 3))
    dtype = c["idx_dtype"]
    dt, ht = G.index_tensors(d, h, where, dtype)
    d2t, _ = G.index_tensors(d2, h, where, dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(device_error=err)
    if path == "staged" and not on_device:
        per_page = sum(p.num_tensors * L * P * p.row_bytes for p in pools)
        kw["staging"] = [torch.empty(2 * per_page, dtype=torch.uint8, device="cuda")
                         for _ in range(2)]
        hpath = hk.HICACHE_PATH_STAGED
    else:
        hpath = hk.HICACHE_PATH_ZERO_COPY
        if path == "single_launch":
            kw["burst_words"] = torch.full((4 * (L + 3),), 7, dtype=torch.int32, device="cuda")
    loc = hk.HICACHE_INDEX_DEVICE if on_device else hk.HICACHE_INDEX_HOST
    opts = hk.Opts(path=hpath, index_location=loc, **kw)
    what = f"seed {seed}: fault {fault}, path {path}, {c}"
    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]

    if on_device:
        hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
        hk.hicache_load_burst(pools, 0, L, ht, d2t, opts=opts,
                              layer_done=[torch.cuda.Event() for _ in range(L)])
        torch.cuda.synchronize()
        assert int(err.item()) == hk.HICACHE_DEVERR_RANGE, what
        for s, p, (dev0, host0) in zip(c["shapes"], pools, imgs):
            keep = np.ones(n, dtype=bool)
            page_rows = s["page_granular"] and s["layout"] == "page_first_direct"
            keep[i:i + P if page_rows else i + 1] = False
            G.oracle_backup(p, dev0, host0, d[keep], h[keep])
            G.assert_host_equal(p, host0, "backup " + what)
            G.oracle_load(p, dev0, host0, range(L), h[keep], d2[keep])
            G.assert_device_equal(p, dev0, "burst " + what)
        return

    if fault != "layer_range":
        with pytest.raises(hk.HiCacheError) as ei:
            hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
        assert ei.value.status == want, what + " / " + ei.value.message
    events = [torch.cuda.Event() for _ in range(max(0, l1 - l0))]
    for e in events:
        e.record()
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pools, l0, l1, ht, d2t, opts=opts, layer_done=events)
    assert ei.value.status == want, what + " / " + ei.value.message
    assert not any(e.query() for e in events), "a layer event was not recorded: " + what
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    assert int(err.item()) == 0, what
    for p, (dev0, host0) in zip(pools, imgs):
        G.assert_host_equal(p, host0, "rejected backup moved bytes: " + what)
        G.assert_device_equal(p, dev0, "rejected burst moved bytes: " + what)
