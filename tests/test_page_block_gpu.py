"""Edge cases of the staged path's page-block copies, bit for bit against the oracle (GPU).

Where a page's device slots are consecutive and the pool is page_first_direct
with 16-byte aligned (page, layer) blocks, the staged gather and scatter move
whole blocks with bulk copies; other pools keep the row kernel.  Each case runs
a staged backup and a staged load-back burst and compares both whole pools with
the oracle.  The cases reach the corners of the block kernel:
  - one CTA (opts.max_ctas = 1) working through thousands of 16 KiB chunks, so
    its chunk tables turn over many times;
  - 16-byte blocks (16-byte rows, page size 1), thousands of one-chunk blocks;
  - 300 layers of K and V, 600 segments: more than one launch holds;
  - a page-granular pool alone (132-byte rows, 8448-byte page blocks);
  - device slots that are consecutive within each page but start off a page
    boundary;
  - shapes that must fall back to the row kernel: 12-byte rows (blocks not
    16-byte aligned) and device slots that are not consecutive within a page.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from tests import gpu_helpers as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _pairs(kind, seed, pages, P, dev_pages, host_pages):
    """Whole host pages in random order; device slots per `kind`."""
    g = np.random.default_rng(seed)
    hp = g.choice(host_pages, size=pages, replace=False)
    h = (hp[:, None] * P + np.arange(P)).reshape(-1)
    if kind == "aligned":
        dp = g.choice(dev_pages, size=pages, replace=False)
        d = (dp[:, None] * P + np.arange(P)).reshape(-1)
    elif kind == "offset":
        # consecutive within each page, starting 3 slots past a page boundary
        dp = g.choice(dev_pages - 1, size=pages, replace=False)
        d = (dp[:, None] * P + 3 + np.arange(P)).reshape(-1)
    else:  # "scattered": device slots random, not consecutive within a page
        d = g.choice(dev_pages * P, size=pages * P, replace=False)
    return d.astype(np.int64), h.astype(np.int64)


CASES = {
    # name: (shape kwargs, pages, device-slot kind, max_ctas, staging pages)
    "one_cta": (dict(L=8, T=2, head_num=4, head_dim=128, dtype_size=2, P=64, slots=64 * 80,
                     pages=80), 40, "aligned", 1, 8),
    "16_byte_blocks": (dict(L=4, T=1, head_num=1, head_dim=8, dtype_size=2, P=1, slots=8192,
                            pages=4096), 3000, "aligned", 0, 1000),
    "600_segments": (dict(L=300, T=2, head_num=1, head_dim=32, dtype_size=2, P=16, slots=16 * 40,
                          pages=40), 20, "aligned", 0, 8),
    "page_granular_alone": (dict(L=4, T=1, head_num=1, head_dim=132, dtype_size=1, P=64,
                                 slots=64 * 128, pages=64, page_granular=True,
                                 value_kind="uint8_uniform"), 40, "aligned", 0, 16),
    "offset_slots": (dict(L=6, T=1, head_num=1, head_dim=576, dtype_size=2, P=64,
                          slots=64 * 200, pages=64), 40, "offset", 0, 16),
    "12_byte_rows": (dict(L=4, T=2, head_num=1, head_dim=6, dtype_size=2, P=16, slots=16 * 128,
                          pages=64), 40, "aligned", 0, 16),
    "scattered_slots": (dict(L=4, T=2, head_num=2, head_dim=64, dtype_size=2, P=16,
                             slots=16 * 128, pages=64), 40, "scattered", 0, 16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_staged_page_blocks_bit_exact(name):
    kw, pages, kind, max_ctas, staging_pages = CASES[name]
    s = G.shape("blk", **kw)
    P = s.page_size
    pool = G.make_pool(s, seed=100 + sorted(CASES).index(name))
    dev_pages = s.device_slots // P
    d, h = _pairs(kind, 7, pages, P, dev_pages, s.host_pages)
    per_page = s.num_tensors * s.num_layers * P * s.row_bytes
    staging = [torch.empty(staging_pages * per_page, dtype=torch.uint8, device="cuda")
               for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    opts = hk.Opts(path=hk.HICACHE_PATH_STAGED, index_location=hk.HICACHE_INDEX_HOST,
                   staging=staging, max_ctas=max_ctas, device_error=err)
    dt, ht = G.index_tensors(d, h, "host")
    dev0, host0 = G.device_images(pool), G.host_images(pool)
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, f"{name}: staged backup")

    # load the host pages back into other device slots of the same kind
    used = np.zeros(s.device_slots, dtype=bool)
    used[d] = True
    g = np.random.default_rng(11)
    if kind == "scattered":
        d2 = g.choice(np.flatnonzero(~used), size=d.size, replace=False).astype(np.int64)
    else:
        free = [p for p in range(dev_pages - (1 if kind == "offset" else 0))
                if not used[p * P:(p + 1) * P + (3 if kind == "offset" else 0)].any()]
        dp2 = g.choice(free, size=pages, replace=False)
        off = 3 if kind == "offset" else 0
        d2 = (dp2[:, None] * P + off + np.arange(P)).reshape(-1).astype(np.int64)
    d2t, _ = G.index_tensors(d2, h, "host")
    dev1 = G.device_images(pool)
    events = [torch.cuda.Event() for _ in range(s.num_layers)]
    hk.hicache_load_burst(pool, 0, s.num_layers, ht, d2t, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    assert all(e.query() for e in events)
    assert int(err.item()) == 0
    G.oracle_load(pool, dev1, host0, range(s.num_layers), h, d2)
    G.assert_device_equal(pool, dev1, f"{name}: staged burst")
