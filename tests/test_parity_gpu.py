"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, bit for bit.

Every test compares whole pools (every byte, touched or not) unless stated.
Sizes span many warp tasks and end in ragged tails; edge cases cover empty
lists, partial pages, 4-byte rows, non-power-of-two page sizes, page-granular
pools, more segments than one launch holds, grid-stride loops, device-located
indices with bad entries, failures that must still record every layer event,
and the full Llama-3-8B-shaped workload in the launch configuration the
benchmark uses.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _opts(path, where, **kw):
    loc = hk.HICACHE_INDEX_DEVICE if where == "device" else hk.HICACHE_INDEX_HOST
    return hk.Opts(path=path, index_location=loc, **kw)


def _staging(nbytes):
    return [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(2)]


def _burst_words(layers):
    """Device words for a single-launch burst (filled with junk: the call zeroes them)."""
    return torch.full((4 * layers,), 12345, dtype=torch.int32, device="cuda")


BURSTS = ["per_layer", "single_launch"]


def _arm(events):
    """Record the events once, then keep the current stream busy for ~0.1 s.

    An event that was never recorded also reports complete, so a test that only
    queries events cannot tell whether a call recorded them.  After _arm, an
    event that a call records on the current stream stays incomplete until the
    sleep ends, and one the call skipped reads complete at once.
    """
    for e in events:
        e.record()
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)


def _assert_recorded_behind_sleep(events):
    assert not any(e.query() for e in events), "a layer event was not recorded by the call"
    torch.cuda.synchronize()
    assert all(e.query() for e in events)


# ---------------------------------------------------------------- tiny MHA pool

def _index_staging(n, dtype=torch.int64):
    bits = 32 if dtype == torch.int32 else 64
    return torch.empty(hk.index_staging_bytes(n, bits), dtype=torch.uint8, device="cuda")


# the staged path plans its copies on the CPU, so it takes host-located indices only
PATH_WHERE = [(p, w) for p in ("zero_copy", "staged", "zero_copy_single_launch")
              for w in ("device", "host", "host_staged_idx")
              if not (p == "staged" and w == "device")]


@pytest.mark.parametrize("path,where", PATH_WHERE)
@pytest.mark.parametrize("dtype", [torch.int32, torch.int64])
def test_tiny_mha_backup_then_load(where, dtype, path):
    """host_staged_idx: host-located indices copied by the library into opts.index_staging."""
    wl = W.tiny_mha()
    s = wl.pools[0]
    extra = {}
    if where == "host_staged_idx":
        where = "host"
        extra["index_staging"] = _index_staging(wl.move_pages * s.page_size, dtype)
    pool = G.make_pool(s, seed=wl.seed)
    d, h, dp, hp = W.page_pairs(wl.seed, wl.move_pages, s.device_slots // s.page_size,
                                s.host_pages, s.page_size)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, where, dtype)
    if path == "staged":
        # room for 5 host pages of all layers: 64 pages take 13 chunks, both buffers alternate
        per_page = s.num_tensors * s.num_layers * s.page_size * s.row_bytes
        opts = _opts(hk.HICACHE_PATH_STAGED, where, staging=_staging(5 * per_page), **extra)
    elif path == "zero_copy_single_launch":
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, where, burst_words=_burst_words(s.num_layers),
                     **extra)
    else:
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, where, **extra)
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "backup")

    # load back into fresh random device pages (distinct from the source pages)
    d2, _, _, _ = W.page_pairs(wl.seed + 100, wl.move_pages, s.device_slots // s.page_size,
                               s.host_pages, s.page_size, exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, where, dtype)
    dev1 = G.device_images(pool)
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    hk.hicache_load_burst(pool, 0, s.num_layers, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.oracle_load(pool, dev1, host0, range(s.num_layers), h, d2)
    G.assert_device_equal(pool, dev1, "load burst")
    # round trip: the fresh slots hold the original rows
    for t in range(s.num_tensors):
        for l in range(s.num_layers):
            a = dev0[t][l].reshape(-1, s.row_bytes)[d]
            b = pool.device_layers[t][l].cpu().numpy().reshape(-1, s.row_bytes)[d2]
            assert np.array_equal(a, b)


# The page counts the pages' unit test probes, then the counts whose staged part
# (a staged backup moves the last quarter of its pages zero-copy, a load the
# last quarter of each layer group's) is 63/64/65/128/129 for the backup and
# 95/96/97 for the load.
@pytest.mark.parametrize("pages", [1, 63, 64, 65, 128, 129, 84, 86, 87, 171, 172, 127, 130])
@pytest.mark.parametrize("path", ["zero_copy", "zero_copy_single_launch", "staged"])
def test_boundary_page_counts(pages, path):
    """The page counts the pages' unit test probes, through the CUDA path.

    The staging buffers hold exactly 64 pages of all layers. A staged backup
    copies all but the last quarter of its pages through them (84/86/87 pages:
    63/64/65 staged, 171/172: 128/129), so those fall just inside, on and just
    past its chunk boundaries. A 3-layer staged load reads its first layer
    zero-copy and copies the other two as one group, in chunks of 96 pages,
    all but the group's last quarter of pages (127/128/130 pages: 95/96/97
    copied).
    """
    s = G.shape(L=3, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=16 * 360, pages=180)
    pool = G.make_pool(s, seed=40 + pages)
    P = s.page_size
    d, h, dp, _ = W.page_pairs(41 + pages, pages, s.device_slots // P, s.host_pages, P)
    where = "host" if path == "staged" else "device"
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, where)
    if path == "staged":
        per_page = s.num_tensors * s.num_layers * P * s.row_bytes
        opts = _opts(hk.HICACHE_PATH_STAGED, where, staging=_staging(64 * per_page))
    elif path == "zero_copy_single_launch":
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, where, burst_words=_burst_words(s.num_layers))
    else:
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, where)
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, f"{pages} pages backup")
    d2, _, _, _ = W.page_pairs(42 + pages, pages, s.device_slots // P, s.host_pages, P,
                               exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, where)
    dev1 = G.device_images(pool)
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    _arm(events)
    hk.hicache_load_burst(pool, 0, s.num_layers, ht, d2t, opts=opts, layer_done=events)
    _assert_recorded_behind_sleep(events)
    G.oracle_load(pool, dev1, host0, range(s.num_layers), h, d2)
    G.assert_device_equal(pool, dev1, f"{pages} pages burst")


@pytest.mark.parametrize("case", ["latent_and_indexer_78_layers", "mha_24_layers"])
def test_staged_burst_with_burst_words(case):
    """A staged burst given burst_words, bit for bit against the oracle.

    Its first layers (one in eight) are read zero-copy: layer 0 with a launch of
    its own, the others as one signalling launch whose events a library stream
    records.  The groups after them go through staging.  The events are checked
    to be recorded by the call, behind a sleep on the caller's stream.  The
    78-layer burst must also stay within a small number of kernel launches:
    one scatter per staging chunk and one zero-copy launch per pool kind and
    layer group, not one launch per layer (beside a kernel that holds the SMs
    every launch waits for room).
    """
    if case == "latent_and_indexer_78_layers":
        lat = G.shape("lat", L=78, T=1, head_num=1, head_dim=576, dtype_size=2, P=64,
                      slots=64 * 48, pages=48)
        idx = G.shape("idx", L=78, T=1, head_num=1, head_dim=132, dtype_size=1, P=64,
                      slots=64 * 48, pages=48, page_granular=True, value_kind="uint8_uniform")
        shapes, pages, staging_mib = [lat, idx], 40, 64
    else:
        shapes, pages, staging_mib = [G.shape("mha", L=24, T=2, head_num=2, head_dim=64,
                                              dtype_size=2, P=16, slots=16 * 96, pages=64)], 30, 16
    pools = [G.make_pool(s, 60 + k) for k, s in enumerate(shapes)]
    s0 = shapes[0]
    L, P = s0.num_layers, s0.page_size
    d, h, _, _ = W.page_pairs(61, pages, s0.device_slots // P, s0.host_pages, P)
    dt, ht = G.index_tensors(d, h, "host")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    opts = _opts(hk.HICACHE_PATH_STAGED, "host", staging=_staging(staging_mib << 20),
                 burst_words=_burst_words(L), device_error=err)
    # a first call in a fresh process loads the kernels it launches, which can
    # take longer than the sleep the events are armed behind
    hk.hicache_load_burst(pools, 0, L, ht, dt, opts=opts)
    torch.cuda.synchronize()
    dev0 = [G.device_images(p) for p in pools]
    host0 = [G.host_images(p) for p in pools]
    events = [torch.cuda.Event() for _ in range(L)]
    _arm(events)
    before = hk.kernel_launches()
    hk.hicache_load_burst(pools, 0, L, ht, dt, opts=opts, layer_done=events)
    launches = hk.kernel_launches() - before
    _assert_recorded_behind_sleep(events)
    assert int(err.item()) == 0
    for p, dv, hs in zip(pools, dev0, host0):
        G.oracle_load(p, dv, hs, range(L), h, d)
        G.assert_device_equal(p, dv, f"{case}: staged burst with burst_words")
    if L == 78:
        # layer 0, one signalling launch for layers 1-9, then four layer groups
        # (4, 16, 28, 20 layers) of one or two chunks each: 15 launches
        assert launches <= 20, f"{launches} kernel launches for one staged burst"


# ------------------------------------------------------ ragged shapes and tails

CASES = [
    # (L, T, head_num, head_dim, dtype_size, P, slots, pages, n, fragmented)
    (3, 2, 1, 6, 2, 3, 300, 70, 157, True),       # 12-byte rows (4-byte path), P=3
    (2, 1, 1, 8, 2, 1, 5000, 4000, 3001, True),    # 16-byte rows, token-random, P=1
    (2, 2, 4, 8, 2, 16, 8192, 600, 4099, True),    # 64-byte rows, ragged final page
    (4, 1, 1, 576, 2, 64, 4096, 80, 64 * 37 + 13, True),  # MLA rows, partial last page
    (2, 2, 8, 128, 2, 64, 8192, 128, 64 * 40, False),     # one contiguous run of 40 pages
    (5, 1, 1, 1024, 2, 256, 4096, 12, 256 * 7 + 100, True),  # P=256
]


@pytest.mark.parametrize("case", CASES, ids=[f"R{c[2]*c[3]*c[4]}_P{c[5]}_n{c[8]}" for c in CASES])
@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("ctas", [0, 16, 32])
def test_ragged_backup_and_load(case, where, ctas):
    """ctas 16: launches of 16 CTAs of 16 warps each, with the deep tasks (about 4 KiB
    each); ctas 32: 8-warp CTAs with the deep tasks."""
    L, T, hn, hd, ds, P, slots, pages, n, frag = case
    s = G.shape(L=L, T=T, head_num=hn, head_dim=hd, dtype_size=ds, P=P, slots=slots, pages=pages)
    pool = G.make_pool(s, seed=n)
    d, h = W.token_pairs(n + 1, n, slots, pages * P, P, fragmented=frag)
    g = np.random.default_rng(n)
    d = d.copy()
    d[g.integers(0, n, size=n // 7)] = d[0]  # backup sources may repeat
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, where)
    hk.hicache_backup_all_layers(pool, dt, ht,
                                 opts=_opts(hk.HICACHE_PATH_ZERO_COPY, where, max_ctas=ctas))
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "backup")
    # load: distinct device destinations, host sources may repeat
    d2 = g.permutation(slots)[:n].astype(np.int64)
    h2 = h.copy()
    h2[g.integers(0, n, size=n // 5)] = h[-1]
    dev1 = G.device_images(pool)
    d2t, h2t = G.index_tensors(d2, h2, where)
    for l in (L - 1, 0):
        hk.hicache_load_layer(pool, l, h2t, d2t,
                              opts=_opts(hk.HICACHE_PATH_ZERO_COPY, where, max_ctas=ctas))
    torch.cuda.synchronize()
    G.oracle_load(pool, dev1, host0, (L - 1, 0), h2, d2)
    G.assert_device_equal(pool, dev1, "load")


@pytest.mark.parametrize("burst", BURSTS)
def test_grid_stride_and_many_segments(burst):
    """Few CTAs loop over many tasks; 600 segments need two launches of the all-layer kernel,
    and a single-launch burst of 280 two-tensor layers is cut into two launches."""
    s = G.shape(L=300, T=2, head_num=1, head_dim=8, dtype_size=2, P=4, slots=256, pages=40)
    pool = G.make_pool(s, seed=5)
    d, h = W.token_pairs(6, 150, 256, 160, 4, fragmented=True)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, "device")
    hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device",
                                                          max_ctas=3))
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "backup 600 segments")
    dev1 = G.device_images(pool)
    words = _burst_words(280) if burst == "single_launch" else None
    events = [torch.cuda.Event() for _ in range(280)]
    hk.hicache_load_burst(pool, 10, 290, ht, dt, layer_done=events,
                          opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device", max_ctas=1,
                                     burst_words=words))
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.oracle_load(pool, dev1, host0, range(10, 290), h, d)
    G.assert_device_equal(pool, dev1, "burst")


@pytest.mark.parametrize("burst", BURSTS)
def test_maximum_layer_count(burst):
    """4096 layers (the most a pool may have) x 2 tensors: 8192 segments, so the backup takes 16
    all-layer launches and the single-launch burst is cut into 16 signalling launches."""
    L = 4096
    s = G.shape(L=L, T=2, head_num=1, head_dim=8, dtype_size=2, P=2, slots=64, pages=16)
    pool = G.make_pool(s, seed=80)
    d, h = W.token_pairs(81, 12, 64, 32, 2, fragmented=True)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, "device")
    hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device"))
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "4096-layer backup")
    d2 = np.setdiff1d(np.arange(64), d)[:12]
    d2t, _ = G.index_tensors(d2, h, "device")
    dev1 = G.device_images(pool)
    words = _burst_words(L) if burst == "single_launch" else None
    events = [torch.cuda.Event() for _ in range(L)]
    hk.hicache_load_burst(pool, 0, L, ht, d2t, layer_done=events,
                          opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device", burst_words=words))
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.oracle_load(pool, dev1, host0, range(L), h, d2)
    G.assert_device_equal(pool, dev1, "4096-layer burst")


def test_maximum_row_size():
    """Rows of 16 MiB (the most a row may hold), page_size 1: 8192 part-tasks per row."""
    s = G.shape(L=2, T=1, head_num=2, head_dim=4 << 20, dtype_size=2, P=1, slots=4, pages=4,
                value_kind="uint8_uniform")
    pool = G.make_pool(s, seed=82)
    d, h = np.array([3, 0], dtype=np.int64), np.array([1, 2], dtype=np.int64)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, "host")
    hk.hicache_backup_all_layers(pool, dt, ht)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "16 MiB rows backup")
    d2, _ = G.index_tensors(np.array([1, 2], dtype=np.int64), h, "host")
    dev1 = G.device_images(pool)
    hk.hicache_load_burst(pool, 0, 2, ht, d2, opts=hk.Opts(burst_words=_burst_words(2)),
                          layer_done=[torch.cuda.Event(), torch.cuda.Event()])
    torch.cuda.synchronize()
    G.oracle_load(pool, dev1, host0, range(2), h, np.array([1, 2], dtype=np.int64))
    G.assert_device_equal(pool, dev1, "16 MiB rows burst")


# ------------------------------------------------------- MLA + DSA indexer pools

def _mla_dsa_shapes(L=5, P=64, pages=24, slots=64 * 40):
    lat = G.shape("mla", L=L, T=1, head_num=1, head_dim=576, dtype_size=2, P=P, slots=slots,
                  pages=pages)
    idx = G.shape("dsa", L=L, T=1, head_num=1, head_dim=132, dtype_size=1, P=P, slots=slots,
                  pages=pages, page_granular=True, value_kind="uint8_uniform")
    return lat, idx


@pytest.mark.parametrize("path", ["zero_copy", "staged", "zero_copy_single_launch"])
def test_two_pools_mla_and_indexer(path):
    lat_s, idx_s = _mla_dsa_shapes()
    pools = [G.make_pool(lat_s, 7), G.make_pool(idx_s, 8)]
    P = lat_s.page_size
    d, h, dp, hp = W.page_pairs(9, 9, lat_s.device_slots // P, lat_s.host_pages, P)
    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]
    dt, ht = G.index_tensors(d, h, "host")
    if path == "staged":
        per_page = sum(p.num_layers * P * p.row_bytes for p in pools)
        opts = _opts(hk.HICACHE_PATH_STAGED, "host", staging=_staging(2 * per_page + 4096))
    elif path == "zero_copy_single_launch":
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host",
                     burst_words=_burst_words(lat_s.num_layers),
                     index_staging=_index_staging(d.size))
    else:
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host")
    hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
    torch.cuda.synchronize()
    for p, (dev0, host0) in zip(pools, imgs):
        G.oracle_backup(p, dev0, host0, d, h)
        G.assert_host_equal(p, host0, "two-pool backup")
    d2, _, _, _ = W.page_pairs(10, 9, lat_s.device_slots // P, lat_s.host_pages, P,
                               exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, "host")
    dev1s = [G.device_images(p) for p in pools]
    events = [torch.cuda.Event() for _ in range(lat_s.num_layers)]
    hk.hicache_load_burst(pools, 0, lat_s.num_layers, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    for p, dev1, (_, host0) in zip(pools, dev1s, imgs):
        G.oracle_load(p, dev1, host0, range(p.num_layers), h, d2)
        G.assert_device_equal(p, dev1, "two-pool burst")


def test_indexer_rejects_partial_pages_on_device():
    """Device-located indices: a page-granular pool skips unaligned pages and flags them."""
    _, idx_s = _mla_dsa_shapes(L=2)
    pool = G.make_pool(idx_s, 11)
    P = idx_s.page_size
    d = np.concatenate([np.arange(P) + 3 * P, np.arange(P) + 5 * P + 1]).astype(np.int64)
    h = np.concatenate([np.arange(P) + 2 * P, np.arange(P) + 7 * P]).astype(np.int64)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dt, ht = G.index_tensors(d, h, "device")
    hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device",
                                                          device_error=err))
    torch.cuda.synchronize()
    assert int(err.item()) == hk.HICACHE_DEVERR_PAGE_ALIGN
    G.oracle_backup(pool, dev0, host0, d[:P], h[:P])  # only the aligned page moves
    G.assert_host_equal(pool, host0, "indexer aligned page only")


# ------------------------------------------------------- page_first host layout

@pytest.mark.parametrize("path,where", [pw for pw in PATH_WHERE if pw[1] != "host_staged_idx"])
def test_page_first_layout_backup_then_load(where, path):
    s = G.shape(L=5, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=4096, pages=96,
                layout="page_first")
    pool = G.make_pool(s, seed=24)
    P = s.page_size
    d, h, dp, _ = W.page_pairs(25, 40, s.device_slots // P, s.host_pages, P)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, where)
    if path == "staged":
        per_page = s.num_tensors * s.num_layers * P * s.row_bytes
        opts = _opts(hk.HICACHE_PATH_STAGED, where, staging=_staging(3 * per_page))
    elif path == "zero_copy_single_launch":
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, where, burst_words=_burst_words(s.num_layers))
    else:
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, where)
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "page_first backup")
    d2, _, _, _ = W.page_pairs(26, 40, s.device_slots // P, s.host_pages, P,
                               exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, where)
    dev1 = G.device_images(pool)
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    hk.hicache_load_burst(pool, 0, s.num_layers, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    G.oracle_load(pool, dev1, host0, range(s.num_layers), h, d2)
    G.assert_device_equal(pool, dev1, "page_first burst")


# (L, T, head_num, head_dim, dtype_size): token-major pools whose rows do not fill
# whole lines take one task per token over its adjacent host layers in the backup
LAYER_ROW_CASES = [
    (1, 1, 1, 66, 2),     # 132-byte rows, a single layer
    (3, 2, 1, 18, 2),     # 36-byte rows
    (78, 1, 1, 132, 1),   # the DSA indexer's token rows
    (130, 1, 2, 36, 2),   # 144-byte rows, two tasks per token (128 + 2 layers)
    (300, 2, 1, 2, 2),    # 4-byte rows; 600 segments: more than one launch holds
]


@pytest.mark.parametrize("case", LAYER_ROW_CASES, ids=[f"L{c[0]}_T{c[1]}_R{c[2]*c[3]*c[4]}"
                                                       for c in LAYER_ROW_CASES])
@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("dtype", [torch.int32, torch.int64])
@pytest.mark.parametrize("order", ["as_allocated", "falling_addresses"])
@pytest.mark.parametrize("ctas", [0, 16])
def test_token_major_backup_by_layer_rows(case, where, dtype, order, ctas):
    """falling_addresses: each tensor's layer buffers sorted so that layer 0 has the
    highest address, which makes every layer's offset from layer 0 negative.  ctas 16:
    launches of 16 CTAs, which take the deep tasks (about 4 KiB of a token's layers)."""
    import dataclasses

    L, T, hn, hd, ds = case
    s = G.shape(L=L, T=T, head_num=hn, head_dim=hd, dtype_size=ds, P=16, slots=1024, pages=48,
                layout="page_first")
    pool = G.make_pool(s, seed=50 + L)
    if order == "falling_addresses":
        pool = dataclasses.replace(pool, device_layers=[
            sorted(per_t, key=lambda b: -b.data_ptr()) for per_t in pool.device_layers])
        assert pool.device_layers[0][0].data_ptr() > pool.device_layers[0][-1].data_ptr() or L == 1
    n = 16 * 20 - 5  # a partial last page
    d, h = W.token_pairs(51 + L, n, s.device_slots, s.host_pages * 16, 16, fragmented=True)
    d = d.copy()
    d[7] = d[3]  # backup sources may repeat
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, where, dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_ZERO_COPY, where,
                                                          device_error=err, max_ctas=ctas))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, f"layer-row backup {case}")


def test_layer_rows_beside_a_direct_pool_and_bad_device_pairs():
    """An MLA latent pool (page_first_direct) and a token-major indexer pool in one
    backup; bad device-located pairs are skipped and flagged in both."""
    lat = G.shape("mla", L=6, T=1, head_num=1, head_dim=576, dtype_size=2, P=64,
                  slots=64 * 32, pages=20)
    idx = G.shape("dsa", L=6, T=1, head_num=1, head_dim=132, dtype_size=1, P=64,
                  slots=64 * 32, pages=20, page_granular=True, value_kind="uint8_uniform",
                  layout="page_first")
    pools = [G.make_pool(lat, 52), G.make_pool(idx, 53)]
    d, h, _, _ = W.page_pairs(54, 9, 32, 20, 64)
    d, h = d.copy(), h.copy()
    d[70] = 64 * 32 + 5  # out of range on the device side
    h[200] = -3          # and on the host side
    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dt, ht = G.index_tensors(d, h, "device")
    hk.hicache_backup_all_layers(pools, dt, ht, opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device",
                                                           device_error=err))
    torch.cuda.synchronize()
    assert int(err.item()) & hk.HICACHE_DEVERR_RANGE
    keep = np.ones(d.size, dtype=bool)
    keep[[70, 200]] = False
    # both pools move token rows here, so exactly the two bad pairs are skipped
    G.oracle_backup(pools[0], imgs[0][0], imgs[0][1], d[keep], h[keep])
    G.assert_host_equal(pools[0], imgs[0][1], "latent pool")
    G.oracle_backup(pools[1], imgs[1][0], imgs[1][1], d[keep], h[keep])
    G.assert_host_equal(pools[1], imgs[1][1], "token-major indexer pool")


# (layout, moved pages, staging in layer blocks of every moved page, layer range).
# Group sizes grow 1, 2, 4, ... while a staging buffer holds every page of the
# group, or chunks of at least 32 pages of it.
STAGED_GROUP_CASES = [
    ("page_first_direct", 24, None, (0, 13)),   # groups 1, 2, 4, 6, one chunk each
    ("page_first_direct", 24, 3, (0, 13)),      # groups 1, 2, 3, 3, 3, 1
    ("page_first_direct", 24, None, (2, 11)),   # groups 1, 2, 6 from layer 2 (tail joins)
    ("page_first", 24, None, (0, 13)),
    ("page_first", 24, 3, (1, 12)),
    # 80 pages, room for 40 pages of 4 layers: groups 1, 2, 4, 5, 1; the group of
    # 4 moves in chunks of 40 + 40 pages, the group of 5 in 32 + 32 + 16
    ("page_first_direct", 80, 2, (0, 13)),
    ("page_first", 80, 2, (0, 13)),
]


@pytest.mark.parametrize("case", STAGED_GROUP_CASES,
                         ids=[f"{c[0]}-n{c[1]}-stage{c[2]}-L{c[3][0]}_{c[3][1]}"
                              for c in STAGED_GROUP_CASES])
def test_staged_load_layer_groups(case):
    """The staged load copies groups of consecutive layers per host page in one DMA."""
    layout, npages, stage_layers, (l0, l1) = case
    s = G.shape(L=13, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=4096, pages=128,
                layout=layout)
    pool = G.make_pool(s, seed=31)
    P = s.page_size
    d, h, dp, _ = W.page_pairs(32, npages, s.device_slots // P, s.host_pages, P)
    dt, ht = G.index_tensors(d, h, "host")
    per_layer = s.num_tensors * npages * P * s.row_bytes  # one layer of every moved page
    layers = stage_layers if stage_layers is not None else s.num_layers
    opts = _opts(hk.HICACHE_PATH_STAGED, "host", staging=_staging(layers * per_layer + 1000))
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    host0 = G.host_images(pool)
    d2, _, _, _ = W.page_pairs(33, npages, s.device_slots // P, s.host_pages, P,
                               exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, "host")
    dev1 = G.device_images(pool)
    events = [torch.cuda.Event() for _ in range(l1 - l0)]
    hk.hicache_load_burst(pool, l0, l1, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.oracle_load(pool, dev1, host0, range(l0, l1), h, d2)
    G.assert_device_equal(pool, dev1, f"staged layer groups {case}")


@pytest.mark.parametrize("path", ["zero_copy", "zero_copy_single_launch", "staged",
                                  "staged_groups"])
def test_mixed_layouts_latent_direct_indexer_token_major(path):
    """Latent pool page_first_direct (16-byte chunks) with an indexer pool in the token-major
    layout (132-byte token rows, 4-byte chunks) in the same calls."""
    lat = G.shape("mla", L=4, T=1, head_num=1, head_dim=576, dtype_size=2, P=64, slots=64 * 32,
                  pages=20)
    idx = G.shape("dsa", L=4, T=1, head_num=1, head_dim=132, dtype_size=1, P=64,
                  slots=64 * 32, pages=20, page_granular=True, value_kind="uint8_uniform",
                  layout="page_first")
    pools = [G.make_pool(lat, 27), G.make_pool(idx, 28)]
    P = 64
    d, h, dp, _ = W.page_pairs(29, 7, 32, 20, P)
    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]
    dt, ht = G.index_tensors(d, h, "host")
    if path.startswith("staged"):
        per_page = sum(p.num_layers * P * p.row_bytes for p in pools)
        # 3 pages of all layers: one-layer loads; 7 pages: every layer of every page
        opts = _opts(hk.HICACHE_PATH_STAGED, "host",
                     staging=_staging((3 if path == "staged" else 7) * per_page))
    elif path == "zero_copy_single_launch":
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host", burst_words=_burst_words(4))
    else:
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host")
    hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
    torch.cuda.synchronize()
    for p, (dev0, host0) in zip(pools, imgs):
        G.oracle_backup(p, dev0, host0, d, h)
        G.assert_host_equal(p, host0, "mixed-layout backup")
    d2, _, _, _ = W.page_pairs(30, 7, 32, 20, P, exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, "host")
    dev1s = [G.device_images(p) for p in pools]
    hk.hicache_load_burst(pools, 0, 4, ht, d2t, opts=opts,
                          layer_done=[torch.cuda.Event() for _ in range(4)])
    torch.cuda.synchronize()
    for p, dev1, (_, host0) in zip(pools, dev1s, imgs):
        G.oracle_load(p, dev1, host0, range(4), h, d2)
        G.assert_device_equal(p, dev1, "mixed-layout burst")


# ------------------------------------------------- hybrid-model state pools (P=1)

@pytest.mark.parametrize("path", ["zero_copy", "zero_copy_single_launch", "staged"])
def test_state_pools_with_multi_mib_rows(path):
    """Mamba-style conv (60 KiB) and SSM (2 MiB) state slots: rows far longer than one warp
    task, split into parts; two pools of different row sizes in one call."""
    conv = G.shape("conv", L=3, T=1, head_num=10240, head_dim=3, dtype_size=2, P=1, slots=16,
                   pages=24)
    ssm = G.shape("ssm", L=3, T=1, head_num=64, head_dim=64 * 128, dtype_size=4, P=1,
                  slots=16, pages=24, value_kind="uint8_uniform")
    pools = [G.make_pool(conv, 70), G.make_pool(ssm, 71)]
    d, h, dp, _ = W.page_pairs(72, 7, 16, 24, 1)
    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]
    dt, ht = G.index_tensors(d, h, "host")
    if path == "staged":
        per_slot = sum(p.num_layers * p.row_bytes for p in pools)
        opts = _opts(hk.HICACHE_PATH_STAGED, "host", staging=_staging(3 * per_slot))
    elif path == "zero_copy_single_launch":
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host", burst_words=_burst_words(3))
    else:
        opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host")
    hk.hicache_backup_all_layers(pools, dt, ht, opts=opts)
    torch.cuda.synchronize()
    for p, (dev0, host0) in zip(pools, imgs):
        G.oracle_backup(p, dev0, host0, d, h)
        G.assert_host_equal(p, host0, "state backup")
    d2, _, _, _ = W.page_pairs(73, 7, 16, 24, 1, exclude_device_pages=dp)
    d2t, _ = G.index_tensors(d2, h, "host")
    dev1s = [G.device_images(p) for p in pools]
    hk.hicache_load_burst(pools, 0, 3, ht, d2t, opts=opts,
                          layer_done=[torch.cuda.Event() for _ in range(3)])
    torch.cuda.synchronize()
    for p, dev1, (_, host0) in zip(pools, dev1s, imgs):
        G.oracle_load(p, dev1, host0, range(3), h, d2)
        G.assert_device_equal(p, dev1, "state burst")


# ------------------------------------------------------- concurrent host threads

@pytest.mark.parametrize("path", ["zero_copy_single_launch", "staged"])
def test_two_threads_burst_concurrently(path):
    """Two host threads, each with its own stream, pool and burst words (or staging
    buffers), run backups and bursts at the same time; both results must match the
    oracle.  The staged buffers hold 2 layers of every page: groups 1, 2, 2, 1."""
    import threading

    s = G.shape("mla", L=6, T=1, head_num=1, head_dim=576, dtype_size=2, P=64, slots=64 * 64,
                pages=48)
    pools = [G.make_pool(s, 40 + k) for k in range(2)]
    P = 64
    pairs = [W.page_pairs(50 + k, 20, 64, 48, P) for k in range(2)]
    fresh = [W.page_pairs(60 + k, 20, 64, 48, P, exclude_device_pages=pairs[k][2])[0]
             for k in range(2)]
    imgs = [(G.device_images(p), G.host_images(p)) for p in pools]
    errors = []

    def work(k):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            d, h = pairs[k][0], pairs[k][1]
            dt, ht = G.index_tensors(d, h, "host")
            d2t, _ = G.index_tensors(fresh[k], h, "host")
            if path == "staged":
                opts = _opts(hk.HICACHE_PATH_STAGED, "host",
                             staging=_staging(2 * d.size * s.row_bytes))
            else:
                opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host", burst_words=_burst_words(6))
            for _ in range(3):
                hk.hicache_backup_all_layers(pools[k], dt, ht, opts=opts, stream=stream)
                hk.hicache_load_burst(pools[k], 0, 6, ht, d2t, opts=opts, stream=stream,
                                      layer_done=[torch.cuda.Event() for _ in range(6)])
            stream.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for k, p in enumerate(pools):
        dev0, host0 = imgs[k]
        d, h = pairs[k][0], pairs[k][1]
        G.oracle_backup(p, dev0, host0, d, h)
        G.assert_host_equal(p, host0, f"thread {k} backup")
        G.oracle_load(p, dev0, host0, range(6), h, fresh[k])
        G.assert_device_equal(p, dev0, f"thread {k} burst")


@pytest.mark.parametrize("burst", BURSTS)
def test_device_indices_written_on_the_stream_are_read_in_order(burst):
    """Device indices written on `stream` just before a call are the ones it uses.

    The index tensors start out as out-of-range sentinels; the real indices are
    copied into them on the stream behind a sleep kernel, right before each
    call.  Reading them any earlier would see the sentinels, skip every pair
    and set the error word.
    """
    s = G.shape(L=5, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=2048, pages=64)
    pool = G.make_pool(s, 44)
    P = s.page_size
    d, h, dp, _ = W.page_pairs(45, 12, s.device_slots // P, s.host_pages, P)
    d2, _, _, _ = W.page_pairs(46, 12, s.device_slots // P, s.host_pages, P,
                               exclude_device_pages=dp)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    real = {k: torch.as_tensor(v).cuda() for k, v in (("d", d), ("h", h), ("d2", d2))}
    idx = {k: torch.full_like(v, -(10 ** 9)) for k, v in real.items()}  # sentinels
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "device", device_error=err,
                 burst_words=_burst_words(s.num_layers) if burst == "single_launch" else None)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(100_000_000)
        idx["d"].copy_(real["d"])
        idx["h"].copy_(real["h"])
        hk.hicache_backup_all_layers(pool, idx["d"], idx["h"], opts=opts, stream=stream)
        torch.cuda._sleep(100_000_000)
        idx["d2"].copy_(real["d2"])
        hk.hicache_load_burst(pool, 0, s.num_layers, idx["h"], idx["d2"], opts=opts,
                              stream=stream,
                              layer_done=[torch.cuda.Event() for _ in range(s.num_layers)])
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "a call read its indices before the stream wrote them"
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "backup")
    G.oracle_load(pool, dev0, host0, range(s.num_layers), h, d2)
    G.assert_device_equal(pool, dev0, "burst")


# ----------------------------------------------------------------- error paths

def test_device_indices_out_of_range_are_skipped_and_flagged():
    s = G.shape(L=2, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=1024, pages=64)
    pool = G.make_pool(s, 12)
    d, h = W.token_pairs(13, 500, 1024, 1024, 16, fragmented=True)
    d = d.copy()
    d[17] = 5000  # out of range
    h = h.copy()
    h[300] = -4
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dt, ht = G.index_tensors(d, h, "device")
    hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device",
                                                          device_error=err))
    torch.cuda.synchronize()
    assert int(err.item()) == hk.HICACHE_DEVERR_RANGE
    keep = np.ones(500, dtype=bool)
    keep[[17, 300]] = False
    G.oracle_backup(pool, dev0, host0, d[keep], h[keep])
    G.assert_host_equal(pool, host0, "skipped bad pairs")


def test_failed_burst_still_records_every_event():
    s = G.shape(L=6, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=1024, pages=64)
    pool = G.make_pool(s, 14)
    d, h = W.token_pairs(15, 64, 1024, 1024, 16, fragmented=True)
    dev0 = G.device_images(pool)
    h = h.copy()
    h[5] = 10 ** 6  # out of range: validation fails on the host
    dt, ht = G.index_tensors(d, h, "host")
    events = [torch.cuda.Event() for _ in range(4)]
    for e in events:
        e.record()
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)  # keep the stream busy so a fresh record is observable
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pool, 1, 5, ht, dt, layer_done=events)
    assert ei.value.status == hk.HICACHE_ERANGE
    assert not any(e.query() for e in events), "events were not re-recorded behind the sleep"
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.assert_device_equal(pool, dev0, "rejected burst moved bytes")


def test_short_index_staging_rejected_and_events_recorded():
    s = G.shape(L=3, T=1, head_num=1, head_dim=64, dtype_size=2, P=4, slots=256, pages=16)
    pool = G.make_pool(s, 21)
    dev0 = G.device_images(pool)
    dt, ht = G.index_tensors(np.arange(8), np.arange(8) + 16, "host")
    events = [torch.cuda.Event() for _ in range(3)]
    for e in events:
        e.record()
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)
    small = torch.empty(hk.index_staging_bytes(8, 64) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pool, 0, 3, ht, dt, layer_done=events,
                              opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "host", index_staging=small))
    assert ei.value.status == hk.HICACHE_EINVAL and "index_staging" in ei.value.message
    assert not any(e.query() for e in events)
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.assert_device_equal(pool, dev0, "rejected burst moved bytes")


def test_short_burst_words_rejected_and_events_recorded():
    s = G.shape(L=4, T=1, head_num=1, head_dim=64, dtype_size=2, P=4, slots=256, pages=16)
    pool = G.make_pool(s, 22)
    dev0 = G.device_images(pool)
    dt, ht = G.index_tensors([1, 2, 3], [5, 6, 7], "device")
    events = [torch.cuda.Event() for _ in range(4)]
    for e in events:
        e.record()
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pool, 0, 4, ht, dt, layer_done=events,
                              opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device",
                                         burst_words=_burst_words(3)))  # 12 words < 16
    assert ei.value.status == hk.HICACHE_EINVAL
    assert not any(e.query() for e in events)
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    G.assert_device_equal(pool, dev0, "rejected burst moved bytes")


def test_single_launch_burst_with_no_rows_completes_events():
    """A page-granular pool with fewer pairs than one page moves nothing; events still fire."""
    _, idx_s = _mla_dsa_shapes(L=3)
    pool = G.make_pool(idx_s, 23)
    dev0 = G.device_images(pool)
    dt, ht = G.index_tensors(np.arange(10), np.arange(10), "device")
    events = [torch.cuda.Event() for _ in range(3)]
    _arm(events)
    hk.hicache_load_burst(pool, 0, 3, ht, dt, layer_done=events,
                          opts=_opts(hk.HICACHE_PATH_ZERO_COPY, "device",
                                     burst_words=_burst_words(3)))
    _assert_recorded_behind_sleep(events)
    G.assert_device_equal(pool, dev0, "no rows")


def test_duplicate_destination_rejected_and_nothing_moves():
    s = G.shape(L=2, T=1, head_num=1, head_dim=64, dtype_size=2, P=4, slots=256, pages=16)
    pool = G.make_pool(s, 16)
    host0 = G.host_images(pool)
    dt, ht = G.index_tensors([1, 2, 3], [5, 6, 5], "host")
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_backup_all_layers(pool, dt, ht)
    assert ei.value.status == hk.HICACHE_EDUP
    torch.cuda.synchronize()
    G.assert_host_equal(pool, host0, "rejected backup moved bytes")


def test_staged_needs_staging_and_whole_pages():
    s = G.shape(L=2, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=1024, pages=64)
    pool = G.make_pool(s, 17)
    d, h = W.token_pairs(18, 40, 1024, 1024, 16, fragmented=True)  # 40 tokens: partial page
    dt, ht = G.index_tensors(d, h, "host")
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_STAGED, "host"))
    assert ei.value.status == hk.HICACHE_ENOSTAGE
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_backup_all_layers(pool, dt, ht, opts=_opts(hk.HICACHE_PATH_STAGED, "host",
                                                              staging=_staging(1 << 20)))
    assert ei.value.status == hk.HICACHE_EINVAL


@pytest.mark.parametrize("fault", ["no_staging", "small_staging", "partial_page"])
def test_failed_staged_burst_still_records_every_event(fault):
    s = G.shape(L=5, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=1024, pages=64)
    pool = G.make_pool(s, 34)
    dev0 = G.device_images(pool)
    P = s.page_size
    d, h, _, _ = W.page_pairs(35, 6, s.device_slots // P, s.host_pages, P)
    if fault == "partial_page":
        d, h = d[:-3], h[:-3]  # the last host page is not whole
    dt, ht = G.index_tensors(d, h, "host")
    staging = {"no_staging": None, "small_staging": _staging(P * s.row_bytes - 16),
               "partial_page": _staging(1 << 20)}[fault]
    events = [torch.cuda.Event() for _ in range(4)]
    _arm(events)
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pool, 1, 5, ht, dt, layer_done=events,
                              opts=_opts(hk.HICACHE_PATH_STAGED, "host", staging=staging))
    assert ei.value.status == (hk.HICACHE_EINVAL if fault == "partial_page"
                               else hk.HICACHE_ENOSTAGE)
    _assert_recorded_behind_sleep(events)
    G.assert_device_equal(pool, dev0, "rejected staged burst moved bytes")


def test_staged_burst_records_every_event_in_groups():
    """Layer groups record one event per layer, each after its own layer's scatter."""
    s = G.shape(L=11, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=2048, pages=64)
    pool = G.make_pool(s, 36)
    P = s.page_size
    d, h, _, _ = W.page_pairs(37, 20, s.device_slots // P, s.host_pages, P)
    dt, ht = G.index_tensors(d, h, "host")
    opts = _opts(hk.HICACHE_PATH_STAGED, "host",
                 staging=_staging(s.num_layers * 20 * P * s.row_bytes * s.num_tensors))
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    host0, dev1 = G.host_images(pool), G.device_images(pool)
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    _arm(events)
    hk.hicache_load_burst(pool, 0, s.num_layers, ht, dt, layer_done=events, opts=opts)
    _assert_recorded_behind_sleep(events)
    G.oracle_load(pool, dev1, host0, range(s.num_layers), h, d)
    G.assert_device_equal(pool, dev1, "staged groups")


BAD_BUFFERS = ["staging_misaligned", "staging_pinned_host", "device_error_misaligned",
               "device_error_pageable", "burst_words_pinned_host", "index_staging_pinned_host"]


@pytest.mark.parametrize("case", BAD_BUFFERS)
def test_bad_gpu_buffers_rejected_and_events_recorded(case):
    """A buffer the GPU would write, of the wrong kind or alignment, is an error status.

    Every case fails host-side validation, so nothing is launched; the load
    still records its events and no byte moves.
    """
    s = G.shape(L=3, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=1024, pages=64)
    pool = G.make_pool(s, 38)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    P = s.page_size
    d, h, _, _ = W.page_pairs(39, 4, s.device_slots // P, s.host_pages, P)
    where = "host" if case.startswith(("staging", "index_staging")) else "device"
    dt, ht = G.index_tensors(d, h, where)
    cuda8 = lambda n: torch.zeros(n, dtype=torch.uint8, device="cuda")  # noqa: E731
    pinned8 = lambda n: torch.zeros(n, dtype=torch.uint8).pin_memory()  # noqa: E731
    kw, want = {}, hk.HICACHE_EINVAL
    path = hk.HICACHE_PATH_ZERO_COPY
    if case == "staging_misaligned":
        path, want = hk.HICACHE_PATH_STAGED, hk.HICACHE_EALIGN
        kw["staging"] = [cuda8(1 << 20)[4:], cuda8(1 << 20)]
    elif case == "staging_pinned_host":
        path = hk.HICACHE_PATH_STAGED
        kw["staging"] = [pinned8(1 << 20), pinned8(1 << 20)]
    elif case == "device_error_misaligned":
        want = hk.HICACHE_EALIGN
        kw["device_error"] = cuda8(8)[2:6]
    elif case == "device_error_pageable":
        kw["device_error"] = torch.zeros(1, dtype=torch.int32)
    elif case == "burst_words_pinned_host":
        kw["burst_words"] = torch.zeros(4 * s.num_layers, dtype=torch.int32).pin_memory()
    else:
        kw["index_staging"] = pinned8(hk.index_staging_bytes(d.size, 64))
    opts = _opts(path, where, **kw)
    with pytest.raises(hk.HiCacheError) as ei:  # every call checks every buffer it is given
        hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    assert ei.value.status == want, ei.value.message
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    _arm(events)
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pool, 0, s.num_layers, ht, dt, opts=opts, layer_done=events)
    assert ei.value.status == want, ei.value.message
    _assert_recorded_behind_sleep(events)
    G.assert_device_equal(pool, dev0, f"{case}: rejected burst moved bytes")
    G.assert_host_equal(pool, host0, f"{case}: rejected backup moved bytes")


def test_host_located_indices_in_device_memory_are_rejected():
    """The CPU validates host-located indices, so they must not be device memory."""
    s = G.shape(L=3, T=1, head_num=1, head_dim=64, dtype_size=2, P=4, slots=256, pages=16)
    pool = G.make_pool(s, 47)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(np.arange(8), np.arange(8) + 16, "device")
    opts = _opts(hk.HICACHE_PATH_ZERO_COPY, "host")  # declared host-located
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    assert ei.value.status == hk.HICACHE_EINVAL and "device memory" in ei.value.message
    events = [torch.cuda.Event() for _ in range(3)]
    _arm(events)
    with pytest.raises(hk.HiCacheError) as ei:
        hk.hicache_load_burst(pool, 0, 3, ht, dt, opts=opts, layer_done=events)
    assert ei.value.status == hk.HICACHE_EINVAL
    _assert_recorded_behind_sleep(events)
    G.assert_device_equal(pool, dev0, "rejected burst moved bytes")
    G.assert_host_equal(pool, host0, "rejected backup moved bytes")


def test_checksum_output_must_be_device_memory():
    s = G.shape(L=2, T=1, head_num=1, head_dim=64, dtype_size=2, P=4, slots=256, pages=16)
    pool = G.make_pool(s, 39)
    dt = torch.arange(8, dtype=torch.int64, device="cuda")
    for out, want in ((torch.zeros(1, dtype=torch.int64).pin_memory(), hk.HICACHE_EINVAL),
                      (torch.zeros(16, dtype=torch.uint8, device="cuda")[4:12], hk.HICACHE_EALIGN)):
        with pytest.raises(hk.HiCacheError) as ei:
            hk.hicache_layer_checksum(pool, 0, 1, dt, out)
        assert ei.value.status == want, ei.value.message


def test_empty_lists_record_events_and_move_nothing():
    s = G.shape(L=3, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=1024, pages=64)
    pool = G.make_pool(s, 19)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(np.zeros(0, np.int64), np.zeros(0, np.int64), "device")
    events = [torch.cuda.Event() for _ in range(3)]
    hk.hicache_backup_all_layers(pool, dt, ht)
    _arm(events)
    hk.hicache_load_burst(pool, 0, 3, ht, dt, layer_done=events)
    _assert_recorded_behind_sleep(events)
    for opts in (_opts(hk.HICACHE_PATH_ZERO_COPY, "device", burst_words=_burst_words(3)),
                 _opts(hk.HICACHE_PATH_STAGED, "host", staging=_staging(1 << 20))):
        loc = "host" if opts.index_location == hk.HICACHE_INDEX_HOST else "device"
        de, he = G.index_tensors(np.zeros(0, np.int64), np.zeros(0, np.int64), loc)
        _arm(events)
        hk.hicache_load_burst(pool, 0, 3, he, de, layer_done=events, opts=opts)
        _assert_recorded_behind_sleep(events)
    G.assert_device_equal(pool, dev0, "empty")
    G.assert_host_equal(pool, host0, "empty")


# ----------------------------------------------------- events gate a consumer

@pytest.mark.parametrize("pages", [256, 8])
@pytest.mark.parametrize("burst", BURSTS + ["staged"])
def test_layer_events_gate_consumer_checksum(burst, pages):
    """A consumer on another stream waits on event l only, and must see layer l fully loaded.

    With 256 pages a layer holds 18.9 MB: the single-launch burst waits for each
    layer's word.  With 8 pages a layer holds 590 KB, so that burst waits once
    per group of 4 layers and records the group's events together; each event
    must still gate its own layer.  The staged variant has room for 4 layers of
    every page, so its layers land in groups.
    """
    s = G.shape("mla", L=12, T=1, head_num=1, head_dim=576, dtype_size=2, P=64, slots=65536,
                pages=512)
    pool = G.make_pool(s, 20)
    d, h, _, _ = W.page_pairs(21, pages, s.device_slots // 64, s.host_pages, 64)
    host0 = G.host_images(pool)
    dt, ht = G.index_tensors(d, h, "device")
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    sums = torch.zeros(s.num_layers, dtype=torch.int64, device="cuda")
    consumer = torch.cuda.Stream()
    load_stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    opts = hk.Opts(burst_words=_burst_words(s.num_layers)) if burst == "single_launch" else None
    ht_load, dt_load = ht, dt
    if burst == "staged":
        dt_load, ht_load = G.index_tensors(d, h, "host")
        opts = _opts(hk.HICACHE_PATH_STAGED, "host",
                     staging=_staging(4 * d.size * s.row_bytes))
    with torch.cuda.stream(load_stream):
        hk.hicache_load_burst(pool, 0, s.num_layers, ht_load, dt_load, layer_done=events,
                              stream=load_stream, opts=opts)
    for l in range(s.num_layers):
        consumer.wait_event(events[l])
        hk.hicache_layer_checksum(pool, 0, l, dt, sums[l:l + 1], stream=consumer)
    torch.cuda.synchronize()
    R = s.row_bytes
    for l in range(s.num_layers):
        blk = host0[0].reshape(s.host_pages, s.num_layers, 64, R)[h // 64, l, h % 64]
        want = int(blk.reshape(-1).view("<u4").astype(np.uint64).sum(dtype=np.uint64))
        assert (int(sums[l].item()) & (2 ** 64 - 1)) == want, f"layer {l} checksum"


# ------------------------------------------- full Llama-3-8B-shaped workload

@pytest.mark.parametrize("burst", BURSTS)
def test_llama3_8b_full_size_backup_and_burst(burst):
    """Full-size pools, the launch configurations the benchmark times; every byte compared."""
    wl = W.llama3_8b_mha()
    s = wl.pools[0]
    P = s.page_size
    pool = G.make_pool(s, wl.seed)
    d, h, dp, hp = W.page_pairs(wl.seed, wl.move_pages, s.device_slots // P, s.host_pages, P)
    d2, _, _, _ = W.page_pairs(wl.seed + 1, wl.move_pages, s.device_slots // P, s.host_pages, P,
                               exclude_device_pages=dp)
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    dt, ht = G.index_tensors(d, h, "device")
    d2t, _ = G.index_tensors(d2, h, "device")
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    opts = hk.Opts(burst_words=_burst_words(s.num_layers)) if burst == "single_launch" else None
    hk.hicache_backup_all_layers(pool, dt, ht)
    hk.hicache_load_burst(pool, 0, s.num_layers, ht, d2t, layer_done=events, opts=opts)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, "full-size backup")
    G.oracle_load(pool, dev0, host0, range(s.num_layers), h, d2)
    G.assert_device_equal(pool, dev0, "full-size burst")
