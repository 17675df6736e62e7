"""Layer-done events must fire while later layers are still loading (GPU).

The per-layer load-back exists so that the attention layer waiting on layer l
can start while layer l+1 is still crossing the link ("[HiCache] Run the
host->device load-back enqueue on a loader thread", Motivation: the inline
path overlapped only about 0.04 % of the copy time, because every copy had
landed before the forward started).  A burst that moved the right bytes but
recorded every event after its last copy would pass every byte comparison, so
these tests time the events themselves.

On a burst of 16 layers of about 18 MiB each, on every load path:
  - the first layer's event completes within twice one layer's share of the
    burst, plus 200 us for launches (the bound the pages imply, read as
    T_burst / L + 20 us, with slack for a shared test box);
  - at least a quarter of the layers complete clearly before the last one (at
    least a fifth of the burst earlier);
  - on the zero-copy paths, which move layers one after another, layer L/2's
    event also completes clearly before layer L-1's;
  - a consumer kernel on another stream, gated only by layer 0's event,
    finishes before the burst's last event.
"""
import pytest

torch = pytest.importorskip("torch")

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as G  # noqa: E402

pytestmark = pytest.mark.gpu

L = 16
PAGES = 256  # 16,384 tokens x 1152 B = 18.9 MB per layer


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hierarchical_kv_cache_gb300.build import build

    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(scope="module")
def pool():
    s = G.shape("mla", L=L, T=1, head_num=1, head_dim=576, dtype_size=2, P=64,
                slots=2 * PAGES * 64, pages=PAGES)
    return G.make_pool(s, 90)


def _timed_burst(pool, path):
    s_pages = pool.device_slots // 64
    d, h, _, _ = W.page_pairs(91, PAGES, s_pages, pool.host_pages, 64)
    if path == "staged":
        dt, ht = G.index_tensors(d, h, "host")
        opts = hk.Opts(path=hk.HICACHE_PATH_STAGED, index_location=hk.HICACHE_INDEX_HOST,
                       staging=[torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
                                for _ in range(2)])
        dev_idx = dt.cuda()
    else:
        dt, ht = G.index_tensors(d, h, "device")
        words = (torch.zeros(4 * L, dtype=torch.int32, device="cuda")
                 if path == "single_launch" else None)
        opts = hk.Opts(path=hk.HICACHE_PATH_ZERO_COPY, index_location=hk.HICACHE_INDEX_DEVICE,
                       burst_words=words)
        dev_idx = dt
    stream = torch.cuda.Stream()
    consumer = torch.cuda.Stream()
    sums = torch.zeros(1, dtype=torch.int64, device="cuda")
    best = None
    for rep in range(3):  # the first run also loads kernels; keep the fastest burst
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(L)]
        done0 = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        hk.hicache_load_burst(pool, 0, L, ht, dt, opts=opts, stream=stream, layer_done=evs)
        consumer.wait_event(evs[0])
        hk.hicache_layer_checksum(pool, 0, 0, dev_idx, sums, stream=consumer)
        done0.record(consumer)
        torch.cuda.synchronize()
        t = [start.elapsed_time(e) for e in evs]
        run = {"t": t, "consumer0": start.elapsed_time(done0)}
        if rep and (best is None or t[-1] < best["t"][-1]):
            best = run
    return best


@pytest.mark.parametrize("path", ["single_launch", "per_layer", "staged"])
def test_layer_events_fire_before_the_burst_ends(pool, path):
    r = _timed_burst(pool, path)
    t = r["t"]
    total = t[-1]
    assert all(t[l] <= t[l + 1] + 1e-3 for l in range(L - 1)), f"events out of order: {t}"
    bound = 2 * total / L + 0.2
    assert t[0] <= bound, f"first event at {t[0]:.3f} ms, bound {bound:.3f} ms (burst {total:.3f})"
    early = sum(1 for l in range(L - 1) if t[l] <= total - 0.2 * total)
    assert early >= L // 4, f"only {early} events clearly before the last: {t}"
    if path != "staged":
        assert t[L // 2] <= total - 0.25 * total, \
            f"layer {L // 2} at {t[L // 2]:.3f} ms, last at {total:.3f} ms"
    assert r["consumer0"] < total, \
        f"consumer of layer 0 finished at {r['consumer0']:.3f} ms, burst ended {total:.3f} ms"
