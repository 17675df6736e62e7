"""Parity at the sweep's own sizes (GPU): the sweep's largest points, bit for bit.

The row-size / page-size / length sweep times up to 262,144 tokens per op.
Bit-exact restoration is the pages' bar ("[HiCache] Opt-in rank-sharded host
tier for DSA under TP", Test: the KV is restored bit-exactly), so these points
are compared with the CPU oracle at those sizes, every byte of both pools,
touched and untouched:
  - 262,144 tokens of 16-byte rows at page size 1, token-random (every pair its
    own run), zero-copy;
  - 262,144 tokens of 2 KiB rows at page size 256, one contiguous run, on the
    zero-copy and the staged path (one 2 GiB DMA span per layer group);
  - 65,536 tokens of 64-byte rows at page size 16, random pages (4,096 DMA
    spans, the most the sweep runs the staged path with at this row size), on
    both paths.
Each case backs up, then overwrites the device pool with other bytes, then
loads the host pages back into the same slots, so a load that did nothing
would leave the wrong bytes.  Pools and pairs are drawn as the sweep draws
them: device and host each hold twice the tokens moved, 4 layers, one tensor.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import pools as hpools  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as G  # noqa: E402

pytestmark = pytest.mark.gpu

LAYERS = 4

# (row bytes, page size, tokens, fragmented, path)
CASES = [
    (16, 1, 262144, True, "zero_copy"),
    (2048, 256, 262144, False, "zero_copy"),
    (2048, 256, 262144, False, "staged"),
    (64, 16, 65536, True, "zero_copy"),
    (64, 16, 65536, True, "staged"),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _ids(c):
    R, P, n, frag, path = c
    return f"R{R}-P{P}-n{n}-{'frag' if frag else 'contig'}-{path}"


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_sweep_point_backup_and_load_bit_exact(case):
    R, P, n, frag, path = case
    slots = 2 * n
    s = W.PoolShape("sweep", num_layers=LAYERS, num_tensors=1, head_num=1, head_dim=R // 2,
                    dtype_size=2, page_size=P, device_slots=slots, host_pages=slots // P,
                    value_kind="uint8_uniform")
    pool = hpools.allocate_pool(s)
    hpools.fill_device_random_(pool, 1000 + n + P, s.value_kind)
    hpools.fill_host_pattern_(pool, salt=R + P)
    torch.cuda.synchronize()
    d, h = W.token_pairs(1000 + n + P, n, slots, slots, P, fragmented=frag)
    runs, full = hk.hicache_plan_runs(d, h, P)
    if path == "staged":
        # the sweep's own eligibility: whole host pages, at most 8192 DMA spans
        assert n % P == 0 and full == n // P and len(runs) <= 8192
        dt, ht = G.index_tensors(d, h, "host")
        staging = [torch.empty(256 << 20, dtype=torch.uint8, device="cuda") for _ in range(2)]
        opts = hk.Opts(path=hk.HICACHE_PATH_STAGED, index_location=hk.HICACHE_INDEX_HOST,
                       staging=staging)
    else:
        dt, ht = G.index_tensors(d, h, "device")
        opts = hk.Opts(path=hk.HICACHE_PATH_ZERO_COPY, index_location=hk.HICACHE_INDEX_DEVICE,
                       burst_words=torch.zeros(4 * LAYERS, dtype=torch.int32, device="cuda"))

    dev0, host0 = G.device_images(pool), G.host_images(pool)
    hk.hicache_backup_all_layers(pool, dt, ht, opts=opts)
    torch.cuda.synchronize()
    G.oracle_backup(pool, dev0, host0, d, h)
    G.assert_host_equal(pool, host0, f"{_ids(case)} backup")

    # other bytes on the device, then the host pages back into the same slots
    hpools.fill_device_random_(pool, 7 + n + P, s.value_kind)
    torch.cuda.synchronize()
    dev1 = G.device_images(pool)
    assert not all(np.array_equal(a, b) for a, b in zip(dev0[0], dev1[0]))
    events = [torch.cuda.Event() for _ in range(LAYERS)]
    hk.hicache_load_burst(pool, 0, LAYERS, ht, dt, opts=opts, layer_done=events)
    torch.cuda.synchronize()
    G.oracle_load(pool, dev1, host0, range(LAYERS), h, d)
    G.assert_device_equal(pool, dev1, f"{_ids(case)} load burst")
    # the restored rows are the rows first backed up
    idx = torch.as_tensor(np.asarray(d, dtype=np.int64))
    for l in range(LAYERS):
        got = pool.device_layers[0][l].view(slots, R).cpu()[idx]
        want = torch.from_numpy(dev0[0][l]).view(slots, R)[idx]
        assert torch.equal(got, want), f"{_ids(case)} layer {l}: round trip"
