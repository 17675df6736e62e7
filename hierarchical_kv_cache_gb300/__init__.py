"""GB300-native paged KV-cache transfer (HiCache backup and per-layer load-back).

The work happens in ``libhicache_gb300.so`` (C ABI in include/hicache.h, CUDA
kernels for sm_103a); this package is its thin Python binding plus pool
allocation helpers.  Build the library with ``hierarchical_kv_cache_gb300.build.build()``.
"""
from ._binding import (  # noqa: F401
    HICACHE_DEVERR_PAGE_ALIGN,
    HICACHE_DEVERR_RANGE,
    HICACHE_DEVERR_TIMEOUT,
    HICACHE_EALIGN,
    HICACHE_ECUDA,
    HICACHE_EDUP,
    HICACHE_EINVAL,
    HICACHE_ENOSTAGE,
    HICACHE_ERANGE,
    HICACHE_INDEX_DEVICE,
    HICACHE_INDEX_HOST,
    HICACHE_LAYOUT_PAGE_FIRST,
    HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP,
    HICACHE_AUTO_STAGED_BELOW_CTAS_LOAD,
    HICACHE_LAYOUT_PAGE_FIRST_DIRECT,
    HICACHE_OP_BACKUP,
    HICACHE_OP_LOAD,
    HICACHE_OK,
    HICACHE_PATH_AUTO,
    HICACHE_PATH_STAGED,
    HICACHE_PATH_ZERO_COPY,
    HiCacheError,
    Opts,
    Pool,
    abi_version,
    hicache_auto_path,
    hicache_backup_all_layers,
    hicache_backup_all_layers_static_staging,
    hicache_check_pairs,
    hicache_layer_checksum,
    hicache_load_burst,
    hicache_load_layer,
    hicache_plan_runs,
    index_staging_bytes,
    kernel_launches,
    lib,
)


def __getattr__(name):
    # torch is only needed for pool allocation; import it on first use so that
    # the binding and the workload generators load without it.
    if name == "allocate_pool":
        from .pools import allocate_pool

        return allocate_pool
    raise AttributeError(name)
