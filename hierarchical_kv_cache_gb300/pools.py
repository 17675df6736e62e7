"""Pool allocation helpers: device layer buffers in HBM, host tensors in pinned memory.

Plumbing only (torch allocates and fills); the transfers themselves go through
the C ABI.  Buffers are raw uint8 tensors because the library moves bytes.
"""
from __future__ import annotations

import torch

from ._binding import HICACHE_LAYOUT_PAGE_FIRST, HICACHE_LAYOUT_PAGE_FIRST_DIRECT, Pool


def allocate_pool(shape, device: str = "cuda", pin_host: bool = True) -> Pool:
    """Allocate an uninitialised pool for a ``workloads.PoolShape``-like object."""
    R = shape.row_bytes
    T, L = shape.num_tensors, shape.num_layers
    dev = [[torch.empty(shape.device_slots * R, dtype=torch.uint8, device=device)
            for _ in range(L)] for _ in range(T)]
    host_bytes = shape.host_pages * L * shape.page_size * R
    host = [torch.empty(host_bytes, dtype=torch.uint8, pin_memory=pin_host) for _ in range(T)]
    return Pool(device_layers=dev, host_tensors=host, num_layers=L, head_num=shape.head_num,
                head_dim=shape.head_dim, dtype_size=shape.dtype_size, page_size=shape.page_size,
                device_slots=shape.device_slots, host_pages=shape.host_pages,
                page_granular=bool(shape.page_granular),
                layout=(HICACHE_LAYOUT_PAGE_FIRST
                        if getattr(shape, "layout", "page_first_direct") == "page_first"
                        else HICACHE_LAYOUT_PAGE_FIRST_DIRECT))


def fill_device_random_(pool: Pool, seed: int, kind: str = "bf16_normal") -> None:
    """Seeded device fill: bf16 ~ N(0,1) or uniform uint8 bytes."""
    g = torch.Generator(device=pool.device_layers[0][0].device)
    g.manual_seed(seed)
    for per_layer in pool.device_layers:
        for buf in per_layer:
            if kind == "bf16_normal":
                v = torch.randn(buf.numel() // 2, generator=g, device=buf.device,
                                dtype=torch.float32).to(torch.bfloat16)
                buf.copy_(v.view(torch.uint8))
            else:
                buf.copy_(torch.randint(0, 256, (buf.numel(),), generator=g, device=buf.device,
                                        dtype=torch.uint8))


def fill_host_pattern_(pool: Pool, salt: int = 0) -> None:
    """Host fill that depends on the byte position (marks untouched bytes).

    A 16 MiB block of position-dependent bytes is laid down repeatedly, each copy
    XORed with its block number, so the fill is cheap even for GiB-sized pools.
    """
    step = 1 << 24
    i = torch.arange(step, dtype=torch.int64)
    base = ((i * 2654435761) >> 11).to(torch.uint8)
    for t, h in enumerate(pool.host_tensors):
        for k, s in enumerate(range(0, h.numel(), step)):
            e = min(h.numel(), s + step)
            h[s:e].copy_(base[:e - s].bitwise_xor((salt + 17 * t + 31 * k) & 0xFF))
