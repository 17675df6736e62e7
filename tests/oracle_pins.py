"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a copy
with a planted mutation) and raises AssertionError when the oracle disagrees
with:

- hand-worked golden images (tests/golden/, derived by hand from the copy
  semantics of the pages' CPU simulation and the page-first layout);
- a restatement of the layout as a numpy array shape [page][layer][token][row]
  with advanced-index assignment (the pages' CPU simulation writes
  dst[dst_indices, layer] = src[src_indices] the same way);
- the round trip: backup then load-back into fresh slots gives back the
  original rows (sglang PR #28434 summary: write back, then load, and check);
- no byte outside the named rows changes (counted, not located by formula);
- pair order does not matter; an empty pair list changes nothing;
- the page counts 1/63/64/65/128/129 that the pages' unit test probes;
- brute force over a tiny pool: every (device slot, host slot) pair alone;
- structural facts of page-first storage read off tagged rows: one host page is
  one contiguous block holding exactly its own tokens for every layer, layer
  blocks in increasing layer order, tokens in increasing in-page order;
- a burst equals its layers loaded one by one, in order;
- for the page_first (token-major) layout: a hand-worked golden image, the
  pages' CPU simulation itself on a [token][layer][row] array, the round trip
  with untouched-byte counts, and token-major structure read off tagged rows.

``run_all_pins`` collects failures instead of stopping at the first, so the
planted-mutation controls can require that every mutant fails some pin.
"""
from __future__ import annotations

import numpy as np

import oracle
from tests import golden_fixtures as gf


def _pool(g, L, P, R, slots, pages, fill="random"):
    dev = [g.integers(0, 256, size=slots * R, dtype=np.uint8) for _ in range(L)]
    host = np.zeros(pages * L * P * R, dtype=np.uint8) if fill == "zero" else \
        g.integers(0, 256, size=pages * L * P * R, dtype=np.uint8)
    return dev, host


def _distinct(g, total, k):
    return g.choice(total, size=k, replace=False).astype(np.int64)


def pin_golden_backup(lib):
    for name in ("backup_L2_P2_R4.txt", "backup_L3_P3_R2.txt"):
        fx = gf.parse(name)
        L, P, R = fx["num_layers"], fx["page_size"], fx["row_bytes"]
        dev = gf.device_image(fx)
        host = np.full(fx["host_pages"] * L * P * R, int(fx["host_fill"], 16), dtype=np.uint8)
        oracle.backup_all_layers(dev, host, fx["device_idx"], fx["host_idx"], page_size=P,
                                 row_bytes=R, lib=lib)
        want = gf.rows_image(fx["expected_host"])
        assert np.array_equal(host, want), f"golden {name}: host image differs"


def pin_golden_load(lib):
    fx = gf.parse("load_L2_P2_R4.txt")
    L, P, R = fx["num_layers"], fx["page_size"], fx["row_bytes"]
    host = gf.rows_image(fx["host_rows"])
    dev = np.full(fx["device_slots"] * R, int(fx["device_fill"], 16), dtype=np.uint8)
    oracle.load_layer(dev, host, fx["layer"], fx["host_idx"], fx["device_idx"], num_layers=L,
                      page_size=P, row_bytes=R, lib=lib)
    want = gf.rows_image(fx["expected_device_layer"])
    assert np.array_equal(dev, want), "golden load: device layer differs"


SHAPES = [  # (L, P, R, device slots, host pages, pairs)
    (1, 1, 4, 16, 16, 7),
    (2, 2, 8, 32, 8, 11),
    (3, 3, 6, 40, 9, 17),
    (4, 4, 16, 64, 16, 40),
    (5, 8, 12, 96, 6, 33),
]


def pin_numpy_shape(lib):
    g = np.random.default_rng(11)
    for (L, P, R, S, H, n) in SHAPES:
        dev, host = _pool(g, L, P, R, S, H)
        d = g.integers(0, S, size=n).astype(np.int64)  # sources may repeat
        h = _distinct(g, H * P, n)
        got = host.copy()
        oracle.backup_all_layers(dev, got, d, h, page_size=P, row_bytes=R, lib=lib)
        want = host.copy().reshape(H, L, P, R)
        for l in range(L):
            want[h // P, l, h % P, :] = dev[l].reshape(S, R)[d]
        assert np.array_equal(got, want.reshape(-1)), f"backup vs numpy shape {(L, P, R)}"
        # load-back of every layer against the same restatement
        dd = _distinct(g, S, n)
        hh = g.integers(0, H * P, size=n).astype(np.int64)
        host4 = host.reshape(H, L, P, R)
        for l in range(L):
            got_l = dev[l].copy()
            oracle.load_layer(got_l, host, l, hh, dd, num_layers=L, page_size=P, row_bytes=R,
                              lib=lib)
            want_l = dev[l].copy().reshape(S, R)
            want_l[dd] = host4[hh // P, l, hh % P, :]
            assert np.array_equal(got_l, want_l.reshape(-1)), f"load vs numpy shape {(L, P, R, l)}"


def pin_exhaustive_single_pairs(lib):
    """Brute force over a tiny pool: every (device slot, host slot) pair alone.

    For each pair the backup must change exactly the R bytes of every layer at
    the [page][layer][token][row] position of that host slot, and the load of
    each layer exactly the device row of that slot; found by comparing whole
    images, not by an address formula.
    """
    L, P, R, S, H = 2, 2, 4, 8, 4
    g = np.random.default_rng(17)
    dev, host = _pool(g, L, P, R, S, H)
    for d in range(S):
        for h in range(H * P):
            got = host.copy()
            oracle.backup_all_layers(dev, got, np.array([d]), np.array([h]), page_size=P,
                                     row_bytes=R, lib=lib)
            want = host.copy().reshape(H, L, P, R)
            for l in range(L):
                want[h // P, l, h % P, :] = dev[l].reshape(S, R)[d]
            assert np.array_equal(got, want.reshape(-1)), f"backup of the single pair {(d, h)}"
            for l in range(L):
                got_l = dev[l].copy()
                oracle.load_layer(got_l, host, l, np.array([h]), np.array([d]), num_layers=L,
                                  page_size=P, row_bytes=R, lib=lib)
                want_l = dev[l].copy().reshape(S, R)
                want_l[d] = host.reshape(H, L, P, R)[h // P, l, h % P]
                assert np.array_equal(got_l, want_l.reshape(-1)), f"load of {(h, d)}, layer {l}"


def pin_round_trip(lib):
    g = np.random.default_rng(12)
    for (L, P, R, S, H, n) in SHAPES:
        dev, host = _pool(g, L, P, R, S, H)
        d = _distinct(g, S, n)
        h = _distinct(g, H * P, n)
        oracle.backup_all_layers(dev, host, d, h, page_size=P, row_bytes=R, lib=lib)
        fresh = [g.integers(0, 256, size=S * R, dtype=np.uint8) for _ in range(L)]
        d2 = _distinct(g, S, n)
        oracle.load_burst(fresh, host, 0, L, h, d2, page_size=P, row_bytes=R, lib=lib)
        for l in range(L):
            a = dev[l].reshape(S, R)[d]
            b = fresh[l].reshape(S, R)[d2]
            assert np.array_equal(a, b), f"round trip layer {l} shape {(L, P, R)}"


def pin_untouched(lib):
    """Exactly n*L*R host bytes change when every device byte differs from the fill."""
    g = np.random.default_rng(13)
    for (L, P, R, S, H, n) in SHAPES:
        dev = [(g.integers(0, 128, size=S * R, dtype=np.uint8) * 2 + 1).astype(np.uint8)
               for _ in range(L)]  # odd bytes
        host = np.zeros(H * L * P * R, dtype=np.uint8)  # even fill
        d = g.integers(0, S, size=n).astype(np.int64)
        h = _distinct(g, H * P, n)
        oracle.backup_all_layers(dev, host, d, h, page_size=P, row_bytes=R, lib=lib)
        assert int(np.count_nonzero(host)) == n * L * R, f"backup changed bytes {(L, P, R)}"
        layer = np.zeros(S * R, dtype=np.uint8)
        src_host = (g.integers(0, 128, size=H * L * P * R, dtype=np.uint8) * 2 + 1).astype(np.uint8)
        dd = _distinct(g, S, n)
        hh = g.integers(0, H * P, size=n).astype(np.int64)
        oracle.load_layer(layer, src_host, L - 1, hh, dd, num_layers=L, page_size=P, row_bytes=R,
                          lib=lib)
        assert int(np.count_nonzero(layer)) == n * R, f"load changed bytes {(L, P, R)}"


def pin_permutation_and_empty(lib):
    g = np.random.default_rng(14)
    for (L, P, R, S, H, n) in SHAPES:
        dev, host = _pool(g, L, P, R, S, H)
        d = g.integers(0, S, size=n).astype(np.int64)
        h = _distinct(g, H * P, n)
        a = host.copy()
        oracle.backup_all_layers(dev, a, d, h, page_size=P, row_bytes=R, lib=lib)
        perm = g.permutation(n)
        b = host.copy()
        oracle.backup_all_layers(dev, b, d[perm], h[perm], page_size=P, row_bytes=R, lib=lib)
        assert np.array_equal(a, b), "pair order changed the backup"
        c = host.copy()
        oracle.backup_all_layers(dev, c, d[:0], h[:0], page_size=P, row_bytes=R, lib=lib)
        assert np.array_equal(c, host), "empty backup changed the host"
        e = dev[0].copy()
        oracle.load_layer(e, host, 0, h[:0], d[:0], num_layers=L, page_size=P, row_bytes=R, lib=lib)
        assert np.array_equal(e, dev[0]), "empty load changed the device"


def pin_boundary_page_counts(lib):
    """Round trip of 1/63/64/65/128/129 whole pages (the page counts the pages' unit test probes)."""
    g = np.random.default_rng(15)
    L, P, R = 2, 4, 8
    S, H = 1024, 160
    for pages in (1, 63, 64, 65, 128, 129):
        dev, host = _pool(g, L, P, R, S, H)
        dp = _distinct(g, S // P, pages)
        hp = _distinct(g, H, pages)
        d = (dp[:, None] * P + np.arange(P)).reshape(-1)
        h = (hp[:, None] * P + np.arange(P)).reshape(-1)
        oracle.backup_all_layers(dev, host, d, h, page_size=P, row_bytes=R, lib=lib)
        fresh = [np.zeros(S * R, dtype=np.uint8) for _ in range(L)]
        oracle.load_burst(fresh, host, 0, L, h, d, page_size=P, row_bytes=R, lib=lib)
        for l in range(L):
            assert np.array_equal(fresh[l].reshape(S, R)[d], dev[l].reshape(S, R)[d]), \
                f"boundary {pages} pages layer {l}"


def _tag_rows(L, S, R):
    """Device rows whose bytes name (layer, slot): u16 layer, u32 slot, then 0x5a padding."""
    assert R >= 8
    layers = []
    for l in range(L):
        rows = np.full((S, R), 0x5A, dtype=np.uint8)
        rows[:, 0:2] = np.frombuffer(np.full(S, l, dtype="<u2").tobytes(), np.uint8).reshape(S, 2)
        rows[:, 2:6] = np.frombuffer(np.arange(S, dtype="<u4").tobytes(), np.uint8).reshape(S, 4)
        layers.append(rows.reshape(-1))
    return layers


def pin_layout_structure(lib):
    """Page-first structure read off tagged rows, without the address formula."""
    g = np.random.default_rng(16)
    for (L, P, H, pages) in ((3, 4, 10, 6), (2, 3, 7, 5), (4, 1, 9, 9)):
        R, S = 8, 64
        dev = _tag_rows(L, S, R)
        host = np.zeros(H * L * P * R, dtype=np.uint8)
        hp = _distinct(g, H, pages)
        # whole host pages; device slots random and distinct
        h = (hp[:, None] * P + np.arange(P)).reshape(-1)
        d = _distinct(g, S, h.size)
        oracle.backup_all_layers(dev, host, d, h, page_size=P, row_bytes=R, lib=lib)
        slot_of_token = dict(zip(h.tolist(), d.tolist()))
        block = L * P * R  # bytes of one host page across all layers
        rows = host.reshape(-1, R)
        for page in range(H):
            blk = rows[page * L * P:(page + 1) * L * P]
            if page not in set(hp.tolist()):
                assert not blk.any(), f"untouched host page {page} was written"
                continue
            lay = blk[:, 0:2].copy().view("<u2").reshape(-1)
            slot = blk[:, 2:6].copy().view("<u4").reshape(-1)
            # every layer appears exactly P times, in non-decreasing order
            assert np.all(np.diff(lay.astype(np.int64)) >= 0), f"layers out of order in page {page}"
            assert sorted(set(lay.tolist())) == list(range(L))
            assert all(int((lay == l).sum()) == P for l in range(L))
            # inside each layer block the slots follow the page's tokens in order
            want = [slot_of_token[page * P + t] for t in range(P)]
            for l in range(L):
                assert slot[lay == l].tolist() == want, f"token order page {page} layer {l}"
        assert host.size == H * block


def pin_burst_is_layer_sequence(lib):
    g = np.random.default_rng(17)
    L, P, R, S, H, n = 5, 4, 12, 48, 8, 20
    dev, host = _pool(g, L, P, R, S, H)
    h = g.integers(0, H * P, size=n).astype(np.int64)
    d = _distinct(g, S, n)
    a = [x.copy() for x in dev]
    oracle.load_burst(a, host, 1, 4, h, d, page_size=P, row_bytes=R, lib=lib)
    b = [x.copy() for x in dev]
    for l in range(1, 4):
        oracle.load_layer(b[l], host, l, h, d, num_layers=L, page_size=P, row_bytes=R, lib=lib)
    for l in range(L):
        assert np.array_equal(a[l], b[l]), f"burst layer {l}"


# ---- page_first host layout: [host token][layer][row] ---------------------

def pin_pf_golden(lib):
    fx = gf.parse("pf_backup_L3_R2.txt")
    L, P, R = fx["num_layers"], fx["page_size"], fx["row_bytes"]
    dev = gf.device_image(fx)
    host = np.full(fx["host_pages"] * P * L * R, int(fx["host_fill"], 16), dtype=np.uint8)
    oracle.pf_backup_all_layers(dev, host, fx["device_idx"], fx["host_idx"], row_bytes=R, lib=lib)
    assert np.array_equal(host, gf.rows_image(fx["expected_host"])), "page_first golden differs"


def pin_pf_numpy_shape(lib):
    """The pages' CPU simulation itself: dst[dst_indices, layer] = src[src_indices]."""
    g = np.random.default_rng(21)
    for (L, P, R, S, H, n) in SHAPES:
        tokens = H * P
        dev, host = _pool(g, L, P, R, S, H)
        d = g.integers(0, S, size=n).astype(np.int64)
        h = _distinct(g, tokens, n)
        got = host.copy()
        oracle.pf_backup_all_layers(dev, got, d, h, row_bytes=R, lib=lib)
        want = host.copy().reshape(tokens, L, R)
        for l in range(L):
            want[h, l] = dev[l].reshape(S, R)[d]
        assert np.array_equal(got, want.reshape(-1)), f"pf backup vs numpy {(L, P, R)}"
        dd = _distinct(g, S, n)
        hh = g.integers(0, tokens, size=n).astype(np.int64)
        host3 = host.reshape(tokens, L, R)
        for l in range(L):
            got_l = dev[l].copy()
            oracle.pf_load_layer(got_l, host, l, hh, dd, num_layers=L, row_bytes=R, lib=lib)
            want_l = dev[l].copy().reshape(S, R)
            want_l[dd] = host3[hh, l]
            assert np.array_equal(got_l, want_l.reshape(-1)), f"pf load vs numpy {(L, P, R, l)}"


def pin_pf_round_trip_and_untouched(lib):
    g = np.random.default_rng(22)
    for (L, P, R, S, H, n) in SHAPES:
        tokens = H * P
        dev = [(g.integers(0, 128, size=S * R, dtype=np.uint8) * 2 + 1).astype(np.uint8)
               for _ in range(L)]
        host = np.zeros(tokens * L * R, dtype=np.uint8)
        d = _distinct(g, S, n)
        h = _distinct(g, tokens, n)
        oracle.pf_backup_all_layers(dev, host, d, h, row_bytes=R, lib=lib)
        assert int(np.count_nonzero(host)) == n * L * R, "pf backup changed bytes"
        fresh = [np.zeros(S * R, dtype=np.uint8) for _ in range(L)]
        d2 = _distinct(g, S, n)
        for l in range(L):
            oracle.pf_load_layer(fresh[l], host, l, h, d2, num_layers=L, row_bytes=R, lib=lib)
            assert int(np.count_nonzero(fresh[l])) == n * R, "pf load changed bytes"
            assert np.array_equal(fresh[l].reshape(S, R)[d2], dev[l].reshape(S, R)[d])


def pin_pf_structure(lib):
    """Token-major storage read off tagged rows: each token holds its L layers in order."""
    g = np.random.default_rng(23)
    L, R, S, tokens, n = 4, 8, 64, 40, 25
    dev = _tag_rows(L, S, R)
    host = np.zeros(tokens * L * R, dtype=np.uint8)
    h = _distinct(g, tokens, n)
    d = _distinct(g, S, n)
    oracle.pf_backup_all_layers(dev, host, d, h, row_bytes=R, lib=lib)
    rows = host.reshape(tokens, L, R)
    slot_of = dict(zip(h.tolist(), d.tolist()))
    for tok in range(tokens):
        blk = rows[tok]
        if tok not in slot_of:
            assert not blk.any(), f"untouched token {tok} written"
            continue
        lay = blk[:, 0:2].copy().view("<u2").reshape(-1).tolist()
        slot = blk[:, 2:6].copy().view("<u4").reshape(-1).tolist()
        assert lay == list(range(L)), f"layers of token {tok} out of order"
        assert slot == [slot_of[tok]] * L, f"token {tok} holds the wrong slot"


PINS = [
    pin_golden_backup,
    pin_golden_load,
    pin_numpy_shape,
    pin_exhaustive_single_pairs,
    pin_round_trip,
    pin_untouched,
    pin_permutation_and_empty,
    pin_boundary_page_counts,
    pin_layout_structure,
    pin_burst_is_layer_sequence,
    pin_pf_golden,
    pin_pf_numpy_shape,
    pin_pf_round_trip_and_untouched,
    pin_pf_structure,
]


def run_all_pins(lib):
    failures = []
    for pin in PINS:
        try:
            pin(lib)
        except Exception as e:  # a mutant may also raise from the wrapper
            failures.append((pin.__name__, repr(e)[:200]))
    return failures
