"""Seeded synthetic workloads for the paged KV-cache transfer.

This module only draws inputs: pool shapes, (device slot, host slot) pair
lists and byte fills.  It holds none of the transfer's arithmetic (no address
or layout computation), so the CPU oracle and the CUDA path can both be fed
from it without sharing any of the method.

Shapes follow the workloads the HiCache pages describe: a Llama-3-8B-shaped MHA
pool, a DeepSeek-V3-shaped MLA latent pool, a 78-layer MLA model with two host
pools (latent KV + DSA indexer-K, "[HiCache] Run the host->device load-back
enqueue on a loader thread", Motivation; "[HiCache] Opt-in rank-sharded host
tier for DSA under TP", Motivation), and a sweep of row sizes, page sizes and
fragmentation.  Device slots of a page-granular allocator are whole pages, so
page lists are drawn as seeded samples of page numbers and expanded to
page_size consecutive token slots.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class PoolShape:
    """Shape of one KV pool (device layer-first, host page-first)."""

    name: str
    num_layers: int
    num_tensors: int  # 2 = K and V, 1 = MLA latent or indexer
    head_num: int
    head_dim: int
    dtype_size: int
    page_size: int
    device_slots: int  # token rows per device layer buffer
    host_pages: int
    page_granular: bool = False
    value_kind: str = "bf16_normal"  # or "uint8_uniform"
    layout: str = "page_first_direct"  # host layout, or "page_first" (token-major)

    @property
    def row_bytes(self) -> int:
        return self.head_num * self.head_dim * self.dtype_size


@dataclass(frozen=True)
class Workload:
    """One transfer workload: pools sharing a pair list and an op description."""

    name: str
    pools: tuple
    move_pages: int  # pages named by the pair list of one op
    seed: int
    description: str = ""
    extra: dict = field(default_factory=dict)


def tiny_mha() -> Workload:
    p = PoolShape("mha", num_layers=4, num_tensors=2, head_num=2, head_dim=64, dtype_size=2,
                  page_size=16, device_slots=4096, host_pages=512)
    return Workload("tiny MHA pool (L=4, 2x64 bf16 K/V, P=16)", (p,), move_pages=64, seed=1,
                    description="back up then load back 64 random distinct pages")


def llama3_8b_mha() -> Workload:
    p = PoolShape("mha", num_layers=32, num_tensors=2, head_num=8, head_dim=128, dtype_size=2,
                  page_size=64, device_slots=65536, host_pages=1024)
    return Workload("Llama-3-8B-shaped MHA pool (L=32, 8x128 bf16 K/V, P=64)", (p,),
                    move_pages=256, seed=2,
                    description="D2H backup of 256 pages, then H2D per-layer load-back of the "
                                "256 pages to fresh random device pages")


def dsv3_mla() -> Workload:
    p = PoolShape("mla", num_layers=61, num_tensors=1, head_num=1, head_dim=576, dtype_size=2,
                  page_size=64, device_slots=65536, host_pages=4096)
    return Workload("DeepSeek-V3-shaped MLA latent pool (L=61, 576 bf16, P=64)", (p,),
                    move_pages=512, seed=3,
                    description="per-layer H2D load-back burst of 512 pages, each layer event "
                                "gating a consumer kernel on that layer")


def mla78_dsa() -> Workload:
    lat = PoolShape("mla", num_layers=78, num_tensors=1, head_num=1, head_dim=576, dtype_size=2,
                    page_size=64, device_slots=131072, host_pages=2048)
    idx = PoolShape("dsa_indexer", num_layers=78, num_tensors=1, head_num=1, head_dim=132,
                    dtype_size=1, page_size=64, device_slots=131072, host_pages=2048,
                    page_granular=True, value_kind="uint8_uniform")
    return Workload("78-layer MLA model with two host pools (latent 1152 B + DSA indexer 132 B "
                    "per token, P=64)", (lat, idx), move_pages=1024, seed=4,
                    description="load-back burst of 1024 pages across both pools with 78 "
                                "layer events, plus an all-layer backup of 1024 pages")


def mamba_state() -> Workload:
    """Hybrid-model state pools: per-request conv and SSM state slots of the Mamba layers.

    The pages list MambaPoolHost among the host pools with staged write-back
    ("[HiCache] Support hybrid-pool staged write-back JIT kernel", implementation
    breakdown) without printing their shapes; these follow a Mamba-2 layer with
    d_inner 4096, 8 groups, d_state 128, d_conv 4 and 64 heads of 64: the conv
    state holds 2*4096 + 2*8*128 = 10240 channels x 3 bf16 taps (60 KiB per slot
    and layer), the SSM state 64 x 64 x 128 fp32 values (2 MiB).  A slot is one
    request, so page_size is 1 and a row is a whole state.
    """
    conv = PoolShape("mamba_conv", num_layers=24, num_tensors=1, head_num=10240, head_dim=3,
                     dtype_size=2, page_size=1, device_slots=64, host_pages=128)
    ssm = PoolShape("mamba_ssm", num_layers=24, num_tensors=1, head_num=64, head_dim=64 * 128,
                    dtype_size=4, page_size=1, device_slots=64, host_pages=128,
                    value_kind="uint8_uniform")
    return Workload("hybrid-model Mamba state pools (24 layers, conv 60 KiB + SSM 2 MiB per "
                    "slot, page_size 1)", (conv, ssm), move_pages=32, seed=5,
                    description="all-layer backup of 32 request slots, then a load-back burst "
                                "of those slots to fresh device slots with 24 layer events")


WORKLOADS = {
    "tiny_mha": tiny_mha,
    "llama3_8b_mha": llama3_8b_mha,
    "dsv3_mla": dsv3_mla,
    "mla78_dsa": mla78_dsa,
    "mamba_state": mamba_state,
}

SWEEP_ROW_BYTES = (16, 64, 256, 1152, 2048)
SWEEP_PAGE_SIZES = (1, 16, 64, 256)
SWEEP_TOKENS = (1024, 4096, 16384, 65536, 262144)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def sample_pages(g: np.random.Generator, total: int, k: int, exclude=None) -> np.ndarray:
    """k distinct page numbers out of range(total), seeded, optionally avoiding ``exclude``."""
    if exclude is None or len(exclude) == 0:
        assert k <= total
        return g.choice(total, size=k, replace=False).astype(np.int64)
    mask = np.ones(total, dtype=bool)
    mask[np.asarray(exclude, dtype=np.int64)] = False
    pool = np.flatnonzero(mask)
    assert k <= pool.size
    return g.choice(pool, size=k, replace=False).astype(np.int64)


def expand_pages(pages: np.ndarray, page_size: int) -> np.ndarray:
    """Token slots of whole pages: page p -> p*page_size .. p*page_size+page_size-1."""
    pages = np.asarray(pages, dtype=np.int64)
    return (pages[:, None] * page_size + np.arange(page_size, dtype=np.int64)[None, :]).reshape(-1)


def page_pairs(seed: int, move_pages: int, device_pages: int, host_pages: int, page_size: int,
               exclude_device_pages=None):
    """(device slots, host slots, device pages, host pages) for move_pages random distinct pages."""
    g = rng(seed)
    dp = sample_pages(g, device_pages, move_pages, exclude_device_pages)
    hp = sample_pages(g, host_pages, move_pages)
    return expand_pages(dp, page_size), expand_pages(hp, page_size), dp, hp


def token_pairs(seed: int, n: int, device_slots: int, host_tokens: int, page_size: int,
                fragmented: bool):
    """Sweep pairs: one contiguous run (page-aligned start) or a seeded random sample.

    Fragmented means random distinct pages (token-random at page_size 1), in a
    random order, for both the device and the host side.
    """
    g = rng(seed)
    if not fragmented:
        d0 = 0
        h0 = 0
        return (np.arange(d0, d0 + n, dtype=np.int64), np.arange(h0, h0 + n, dtype=np.int64))
    pages = -(-n // page_size)
    dp = sample_pages(g, device_slots // page_size, pages)
    hp = sample_pages(g, host_tokens // page_size, pages)
    return expand_pages(dp, page_size)[:n], expand_pages(hp, page_size)[:n]


def random_bytes(seed: int, nbytes: int, kind: str = "uint8_uniform") -> np.ndarray:
    """Seeded fill: uint8 uniform, or bf16 ~ N(0,1) (upper half of an fp32 normal)."""
    g = rng(seed)
    if kind == "uint8_uniform":
        return g.integers(0, 256, size=nbytes, dtype=np.uint8)
    assert kind == "bf16_normal" and nbytes % 2 == 0
    f = g.standard_normal(nbytes // 2, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8)


def sentinel_bytes(nbytes: int, salt: int = 0) -> np.ndarray:
    """A fill that is a fixed function of the byte position: marks untouched bytes."""
    i = np.arange(nbytes, dtype=np.uint64)
    return (((i * np.uint64(2654435761)) >> np.uint64(11)) ^ np.uint64(salt)).astype(np.uint8)
