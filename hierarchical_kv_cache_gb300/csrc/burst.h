// burst.h -- the single-launch load-back burst (see burst.cu).
#pragma once

#include <vector>

#include "hicache_internal.h"

namespace hk {

constexpr int kBurstWordsPerLayer = 4;

// True when the driver provides the stream memory wait the burst relies on.
bool signaled_burst_available();

// Loads layers [layer_begin, layer_end) of every pool in one launch and records
// evs[l - layer_begin] once layer l has landed; o.burst_words holds at least
// kBurstWordsPerLayer * (layer_end - layer_begin) device words.  Every event is recorded on every
// return path.
hicache_status signaled_burst(const std::vector<PoolInfo>& pools, const SideSpec& side,
                              const IndexSet& idx, const hicache_opts& o, int32_t layer_begin,
                              int32_t layer_end, cudaStream_t stream, cudaEvent_t* evs);

}  // namespace hk
