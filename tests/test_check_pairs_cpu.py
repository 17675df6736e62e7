"""hicache_check_pairs (host index validation) against the rules written out pair by pair.

The library validates a pair list in one pass over its runs (stretches where
both indices step by one), checking ranges at run ends, marking destinations a
bitmap word at a time and reading the page structure off the run starts.  The
reference below applies the same rules the plain way, to every pair, and the
two must agree on the status and on the pair the error message names, over
random lists built to hit every rule: long runs and single pairs, repeated
destinations, values out of range on either side (negative, past the pool,
near the int64 limits and wrapping past the largest int64), int32 and int64
indices, and page-granular pools with whole or broken pages.
No GPU and no CUDA call is involved.
"""
import ctypes
import re

import numpy as np
import pytest

import hierarchical_kv_cache_gb300 as hk
from hierarchical_kv_cache_gb300 import _binding as B
from hierarchical_kv_cache_gb300.build import build
from tests.test_abi_cpu import c_pool

I64_MAX = np.iinfo(np.int64).max
I64_MIN = np.iinfo(np.int64).min


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def reference(pools, d, h, dest_is_device):
    """(status, pair or page named by the message) from the rules, pair by pair."""
    d = [int(x) for x in d]
    h = [int(x) for x in h]
    n = len(d)
    dev_lim = min(p["slots"] for p in pools)
    host_lim = min(p["pages"] * p["P"] for p in pools)
    for i in range(n):
        if not 0 <= d[i] < dev_lim or not 0 <= h[i] < host_lim:
            return hk.HICACHE_ERANGE, i
    dst = d if dest_is_device else h
    seen = set()
    for i, x in enumerate(dst):
        if x in seen:
            return hk.HICACHE_EDUP, i
        seen.add(x)
    if any(p["granular"] for p in pools):
        P = pools[0]["P"]
        if n % P:
            return hk.HICACHE_EINVAL, None
        for k in range(0, n, P):
            if d[k] % P or h[k] % P:
                return hk.HICACHE_EINVAL, k
            if any(d[k + t] != d[k] + t or h[k + t] != h[k] + t for t in range(P)):
                return hk.HICACHE_EINVAL, k
    return hk.HICACHE_OK, None


def call(pools, d, h, dest_is_device, dtype):
    arr = (B.c_pool * len(pools))(*[c_pool(L=2, T=1, P=p["P"], slots=p["slots"], pages=p["pages"],
                                           page_granular=int(p["granular"])) for p in pools])
    d = np.ascontiguousarray(d, dtype=dtype)
    h = np.ascontiguousarray(h, dtype=dtype)
    bits = 32 if dtype == np.int32 else 64
    st = B.lib().hicache_check_pairs(arr, len(pools), d.ctypes.data, h.ctypes.data, bits, d.size,
                                     int(dest_is_device))
    return st, B.lib().hicache_last_error().decode()


def named(status, message):
    """The pair (or page start) an error message names."""
    if status == hk.HICACHE_ERANGE:
        return int(re.search(r"at pair (\d+)", message).group(1))
    if status == hk.HICACHE_EDUP:
        return int(re.search(r"second time at pair (\d+)", message).group(1))
    m = re.search(r"pairs? (\d+)", message)
    return int(m.group(1)) if m else None


def random_list(g, P, slots, host_tokens, granular, dtype):
    """Distinct whole pages on both sides (sorted half the time, so that runs span
    several pages), sometimes cut inside the last page, and in most lists one
    planted fault."""
    kd, kh = slots // P, host_tokens // P
    k = int(g.integers(0, min(kd, kh, 1500 // P + 1) + 1))
    sort = g.random() < 0.5

    def pages(total):
        x = g.choice(total, size=k, replace=False).astype(np.int64)
        return np.sort(x) if sort else x

    d = (pages(kd)[:, None] * P + np.arange(P)).reshape(-1)
    h = (pages(kh)[:, None] * P + np.arange(P)).reshape(-1)
    if not granular and d.size and g.random() < 0.4:
        cut = int(g.integers(1, d.size + 1))
        d, h = d[:cut], h[:cut]
    n = d.size
    if n and g.random() < 0.7:
        fault = int(g.integers(0, 6))
        i = int(g.integers(0, n))
        big = I64_MAX if dtype == np.int64 else np.iinfo(np.int32).max
        small = I64_MIN if dtype == np.int64 else np.iinfo(np.int32).min
        side, lim = (d, slots) if g.random() < 0.5 else (h, host_tokens)
        if fault == 0:
            side[i] = -1 - int(g.integers(0, 5))
        elif fault == 1:
            side[i] = lim + int(g.integers(0, 5))
        elif fault == 2:
            side[i] = big
        elif fault == 3:  # a run that steps past the largest value and wraps
            side[i] = big
            if i + 1 < n:
                side[i + 1] = small
        elif fault == 4 and n > 1:  # a destination (or source) named twice
            side[i] = side[(i + 1 + int(g.integers(0, n - 1))) % n]
        elif fault == 5:  # one pair shifted: breaks its page, may collide
            side[i] = (side[i] + 1) % lim
    return d, h


CONFIGS = [(1, False), (2, False), (3, False), (16, False), (64, False), (4, True), (16, True),
           (64, True)]


@pytest.mark.parametrize("P,granular", CONFIGS)
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
@pytest.mark.parametrize("dest_is_device", [False, True])
def test_check_pairs_matches_the_rules(P, granular, dtype, dest_is_device):
    g = np.random.default_rng(P * 1000 + granular * 100 + (dtype == np.int64) * 10 + dest_is_device)
    for trial in range(60):
        slots = P * int(g.integers(2, 200))
        pages = int(g.integers(2, 200))
        pools = [dict(P=P, slots=slots, pages=pages, granular=granular)]
        if g.random() < 0.3:  # a second pool with other limits
            pools.append(dict(P=P, slots=P * int(g.integers(2, 200)), pages=int(g.integers(2, 200)),
                              granular=bool(g.random() < 0.5) if P > 1 else False))
        d, h = random_list(g, P, slots, pages * P, granular, dtype)
        want, where = reference(pools, d, h, dest_is_device)
        got, msg = call(pools, d, h, dest_is_device, dtype)
        ctx = f"trial {trial}: n={d.size} pools={pools} message={msg!r}"
        assert got == want, ctx
        if want in (hk.HICACHE_ERANGE, hk.HICACHE_EDUP) or (want == hk.HICACHE_EINVAL and where is not None):
            assert named(got, msg) == where, ctx


def test_check_pairs_edges():
    pools = [dict(P=4, slots=64, pages=8, granular=False)]
    ok = (hk.HICACHE_OK, "")
    assert call(pools, [], [], True, np.int64) == ok
    assert call(pools, [63], [31], True, np.int64) == ok
    # a run that wraps past the largest int64 is out of range, not a long run
    st, _ = call(pools, [I64_MAX, I64_MIN], [0, 1], True, np.int64)
    assert st == hk.HICACHE_ERANGE
    # a range error outranks an earlier duplicate
    st, msg = call(pools, [5, 5, 64], [0, 1, 2], True, np.int64)
    assert st == hk.HICACHE_ERANGE and "at pair 2" in msg
    # the duplicate found inside a run is the first repeated pair
    st, msg = call(pools, list(range(10, 20)) + list(range(15, 18)), list(range(13)), True, np.int64)
    assert st == hk.HICACHE_EDUP and "at pair 10" in msg and "destination 15" in msg
    # destinations are host slots for a backup and device slots for a load
    assert call(pools, [1, 1], [2, 3], False, np.int64)[0] == hk.HICACHE_OK
    assert call(pools, [1, 1], [2, 3], True, np.int64)[0] == hk.HICACHE_EDUP
    with pytest.raises(hk.HiCacheError):
        hk.hicache_check_pairs([], [1], [2], dest_is_device=True)  # no pools
    with pytest.raises(TypeError):
        hk.hicache_check_pairs([], np.array([1], np.int32), np.array([2], np.int64),
                               dest_is_device=True)


def test_check_pairs_runs_of_every_alignment():
    """Runs that start and end at every offset inside a bitmap word, on both sides."""
    pools = [dict(P=1, slots=1024, pages=1024, granular=False)]
    for start in range(0, 130, 7):
        for ln in (1, 2, 63, 64, 65, 127, 128, 129, 200):
            if start + ln > 1024:
                continue
            d = np.arange(start, start + ln)
            h = np.arange(ln)  # both sides step by one: a single run
            assert call(pools, d, h, True, np.int64)[0] == hk.HICACHE_OK
            # the last destination once more, as a run of its own
            st, msg = call(pools, np.r_[d, d[-1]], np.r_[h, ln + 3], True, np.int64)
            assert st == hk.HICACHE_EDUP and f"at pair {ln}" in msg, (start, ln, msg)
            # a later run overlapping an earlier one from its middle on
            if ln >= 4:
                d3 = np.r_[d, np.arange(start + ln // 2, start + ln + 5)]
                h3 = np.r_[h, np.arange(ln + 10, ln + 10 + d3.size - ln)]
                st, msg = call(pools, d3, h3, True, np.int64)
                assert st == hk.HICACHE_EDUP and f"at pair {ln}" in msg, (start, ln, msg)
    # two calls in a row on one thread: the bitmap was left clear
    assert call(pools, np.arange(100), np.arange(100), True, np.int64)[0] == hk.HICACHE_OK
    assert call(pools, np.arange(100), np.arange(100), True, np.int64)[0] == hk.HICACHE_OK


def test_check_pairs_is_exported_with_its_wrapper():
    assert hasattr(ctypes.CDLL(B.LIB_PATH), "hicache_check_pairs")
    assert hk.hicache_check_pairs is B.hicache_check_pairs
