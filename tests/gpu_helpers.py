"""Helpers shared by the GPU parity tests: pool images and oracle runs.

The CUDA path runs through the C ABI (the package binding); the expected
bytes come from the CPU oracle applied to numpy copies of the same pools taken
before the transfer.  The two share nothing but the seeded input generators.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from hierarchical_kv_cache_gb300 import pools as hpools
from hierarchical_kv_cache_gb300.workloads import PoolShape


def shape(name="p", L=4, T=2, head_num=2, head_dim=64, dtype_size=2, P=16, slots=4096, pages=512,
          page_granular=False, value_kind="bf16_normal", layout="page_first_direct"):
    return PoolShape(name, num_layers=L, num_tensors=T, head_num=head_num, head_dim=head_dim,
                     dtype_size=dtype_size, page_size=P, device_slots=slots, host_pages=pages,
                     page_granular=page_granular, value_kind=value_kind, layout=layout)


def make_pool(s: PoolShape, seed: int):
    pool = hpools.allocate_pool(s)
    hpools.fill_device_random_(pool, seed, s.value_kind)
    hpools.fill_host_pattern_(pool, salt=seed)
    torch.cuda.synchronize()
    return pool


def device_images(pool):
    return [[buf.cpu().numpy().copy() for buf in per_layer] for per_layer in pool.device_layers]


def host_images(pool):
    return [h.numpy().copy() for h in pool.host_tensors]


def oracle_backup(pool, dev_imgs, host_imgs, d, h):
    for t in range(pool.num_tensors):
        if pool.layout == 1:  # page_first, token-major
            oracle.pf_backup_all_layers(dev_imgs[t], host_imgs[t], d, h, row_bytes=pool.row_bytes)
        else:
            oracle.backup_all_layers(dev_imgs[t], host_imgs[t], d, h, page_size=pool.page_size,
                                     row_bytes=pool.row_bytes)


def oracle_load(pool, dev_imgs, host_imgs, layers, h, d):
    for t in range(pool.num_tensors):
        for l in layers:
            if pool.layout == 1:
                oracle.pf_load_layer(dev_imgs[t][l], host_imgs[t], l, h, d,
                                     num_layers=pool.num_layers, row_bytes=pool.row_bytes)
            else:
                oracle.load_layer(dev_imgs[t][l], host_imgs[t], l, h, d,
                                  num_layers=pool.num_layers, page_size=pool.page_size,
                                  row_bytes=pool.row_bytes)


def assert_host_equal(pool, want_imgs, what=""):
    for t, h in enumerate(pool.host_tensors):
        got = h.numpy()
        if not np.array_equal(got, want_imgs[t]):
            bad = np.flatnonzero(got != want_imgs[t])
            raise AssertionError(f"{what}: host tensor {t} differs at {bad.size} bytes, first {bad[:8]}")


def assert_device_equal(pool, want_imgs, what="", layers=None):
    for t in range(pool.num_tensors):
        for l in (layers if layers is not None else range(pool.num_layers)):
            got = pool.device_layers[t][l].cpu().numpy()
            if not np.array_equal(got, want_imgs[t][l]):
                bad = np.flatnonzero(got != want_imgs[t][l])
                raise AssertionError(f"{what}: device tensor {t} layer {l} differs at {bad.size} "
                                     f"bytes, first {bad[:8]}")


def index_tensors(d, h, where: str, dtype=torch.int64):
    """Index tensors on the device, or in pinned host memory."""
    dt = torch.as_tensor(np.asarray(d), dtype=dtype)
    ht = torch.as_tensor(np.asarray(h), dtype=dtype)
    if where == "device":
        return dt.cuda(), ht.cuda()
    return dt.pin_memory(), ht.pin_memory()
