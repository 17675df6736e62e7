// staged.h -- the staged transfer path and the path chooser.
#pragma once

#include <vector>

#include "hicache_internal.h"

namespace hk {

// All-layer backup through HBM staging: a gather kernel packs chunks of whole
// host pages into a page-first staging buffer, then one copy-engine DMA per run
// of consecutive host pages (per tensor) writes them to the host pool; two
// staging buffers alternate so the gather of chunk k+1 overlaps the DMA of k.
hicache_status staged_backup(const std::vector<PoolInfo>& pools, const hicache_opts& o,
                             const IndexSet& idx, cudaStream_t stream);

// Load-back through HBM staging: after the first layers (read zero-copy), per
// group of consecutive layers, 2-D DMAs of the group's blocks of every host
// page run into staging and one scatter kernel per staging chunk into the
// device slots; layer_done[l - layer_begin] is recorded once layer l's group
// has landed.
hicache_status staged_load(const std::vector<PoolInfo>& pools, const hicache_opts& o,
                           const IndexSet& idx, int32_t layer_begin, int32_t layer_end,
                           cudaStream_t stream, cudaEvent_t* layer_done);

// Creates, once per calling thread and current device, the copy stream and
// events the staged path uses (later calls find them ready).
hicache_status staged_resources_ready();

// AUTO path choice for one call that moves `layers` layers (see
// hicache_auto_path in hicache.h for the rule).
hicache_path choose_path(const std::vector<PoolInfo>& pools, const hicache_opts& o,
                         const IndexSet& idx, Dir dir, int32_t layers);

// Host page of each group of page_size pairs when the pairs are whole aligned
// host pages in groups (pairs kP..kP+P-1 are host tokens p*P..p*P+P-1);
// returns false otherwise.
bool host_page_groups(const void* host_idx, int32_t bits, int64_t n, int32_t page_size,
                      std::vector<int64_t>* pages);

}  // namespace hk
