// burst.h -- the single-launch load-back burst (see burst.cu).
#pragma once

#include <vector>

#include "hicache_internal.h"

namespace hk {

constexpr int kBurstWordsPerLayer = 4;

// Bytes of one layer (all pools) from which the first layer of a burst gets a
// launch of its own.  Below it the whole burst is one signalling launch: on
// GB300 a 4-layer burst of 4 MiB layers moved 166 GB/s with the extra launch
// (about 20 us of fixed cost per burst).
constexpr int64_t kSplitFirstLayerBytes = int64_t(16) << 20;

// Layers of a signalling launch are counted and waited for in groups of at
// least this many bytes (all pools): the kernel sets one word per group once
// the group's layers have landed, and the group's events are recorded
// together after one stream wait.  Each stream memory wait costs the host
// about 0.6 us to enqueue, which a burst of small layers would otherwise pay
// per layer (89 against 30 us of host time for a one-page 78-layer burst).
// Layers of this size or more are groups of their own, so each layer's event
// comes as soon as it lands.
constexpr int64_t kSignalGroupBytes = int64_t(2) << 20;

// True when the driver provides the stream memory wait the burst relies on.
bool signaled_burst_available();

// Loads layers [layer_begin, layer_end) of every pool in one signalling launch
// (two when a layer holds kSplitFirstLayerBytes or more: the first layer alone,
// then the rest) and records
// evs[l - layer_begin] once layer l has landed; o.burst_words holds at least
// kBurstWordsPerLayer * (layer_end - layer_begin) device words.  Every event is recorded on every
// return path.
hicache_status signaled_burst(const std::vector<PoolInfo>& pools, const SideSpec& side,
                              const IndexSet& idx, const hicache_opts& o, int32_t layer_begin,
                              int32_t layer_end, cudaStream_t stream, cudaEvent_t* evs);

}  // namespace hk
