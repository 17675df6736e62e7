"""Child process of tests/test_zz_no_alloc.py: device memory around the
allocation-free backup entry point, measured in a fresh process.

Prints one JSON line: the device's free memory and torch's reserved memory
after a warm-up call with no pairs and after two calls that move pages, and
whether the moved host pages hold the device bytes (checked here against the
device pool itself, through plain torch indexing of the page-first layout).
"""
import json
import os
import sys

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, REPO)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import hierarchical_kv_cache_gb300 as hk  # noqa: E402
from hierarchical_kv_cache_gb300 import pools as hpools  # noqa: E402
from hierarchical_kv_cache_gb300 import workloads as W  # noqa: E402
from hierarchical_kv_cache_gb300.build import build  # noqa: E402


def main():
    build()
    torch.cuda.set_device(0)
    s = W.PoolShape("mha", num_layers=8, num_tensors=2, head_num=4, head_dim=128,
                    dtype_size=1, page_size=64, device_slots=64 * 96, host_pages=80)
    P, L, R = s.page_size, s.num_layers, s.row_bytes
    pool = hpools.allocate_pool(s)
    hpools.fill_device_random_(pool, 7, s.value_kind)
    hpools.fill_host_pattern_(pool, salt=7)
    lists = []
    for call in range(2):
        d, h, dp, hp = W.page_pairs(60 + call, 70, s.device_slots // P, s.host_pages, P)
        lists.append((torch.as_tensor(d).pin_memory(), torch.as_tensor(h).pin_memory(), dp, hp))
    empty = torch.empty(0, dtype=torch.int64).pin_memory()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    hk.hicache_backup_all_layers_static_staging(pool, empty, empty, stream=stream)  # warm-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    res0 = torch.cuda.memory_reserved()
    for d, h, _, _ in lists:
        hk.hicache_backup_all_layers_static_staging(pool, d, h, stream=stream)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    res1 = torch.cuda.memory_reserved()
    # the second list's pages: host page hp[k] holds, for every layer, device page dp[k]
    _, _, dp, hp = lists[1]
    ok = True
    for t in range(s.num_tensors):
        host = pool.host_tensors[t].view(s.host_pages, L, P * R)
        for l in range(L):
            dev = pool.device_layers[t][l].view(s.device_slots // P, P * R).cpu()
            ok = ok and torch.equal(host[torch.as_tensor(hp), l], dev[torch.as_tensor(dp)])
    print(json.dumps({"free_before_warm_up": free_before, "free_after_warm_up": free0,
                      "free_after_calls": free1, "warm_up_took": free_before - free0,
                      "torch_reserved_after_warm_up": res0, "torch_reserved_after_calls": res1,
                      "moved_ok": bool(ok),
                      "module_loading": os.environ.get("CUDA_MODULE_LOADING")}), flush=True)


if __name__ == "__main__":
    main()
