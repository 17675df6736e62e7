// burst.cu -- the single-launch load-back burst with per-layer events.
//
// The per-layer load-back of "[HiCache] Run the host->device load-back enqueue
// on a loader thread" signals a layer-done event after each layer so that the
// attention layer waiting on it can start early.  Launching one kernel per
// layer pays a launch gap plus a ramp-up and a drain per layer.  Here one
// launch of the row-copy kernel covers every layer of the burst (tasks in
// layer order); the warp that completes a layer sets that layer's word in
// device memory.  A library stream, forked from the caller's stream before the
// launch, waits on each word in turn with a stream memory wait (handled by the
// GPU front end, not by a spinning kernel) and records the caller's event for
// that layer.  The caller's stream joins the library stream before the call
// returns, so the whole burst stays ordered on the caller's stream.
//
// No wait can outlive the launch: the waits are enqueued only after the launch
// succeeded, and the last CTA to leave the launch sets every word of its layers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "burst.h"

namespace hk {

namespace {

using WaitValue32Fn = CUresult(CUDAAPI*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

hicache_status cuda_fail(cudaError_t e, const std::string& what) {
  return fail(HICACHE_ECUDA, what + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

// Library stream and events of the burst, created once per thread and device.
struct BurstRes {
  bool init = false;
  cudaStream_t sig = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

WaitValue32Fn wait_value32() {
  static std::once_flag once;
  static WaitValue32Fn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WaitValue32Fn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

hicache_status get_res(BurstRes** out) {
  static thread_local BurstRes res[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(HICACHE_EINVAL, "device ordinal above 63");
  BurstRes& r = res[dev];
  if (!r.init) {
    e = cudaStreamCreateWithFlags(&r.sig, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreate(burst signal stream)");
    e = cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate(burst)");
    r.init = true;
  }
  *out = &r;
  return HICACHE_OK;
}

void record_from(cudaEvent_t* evs, int32_t from, int32_t count, cudaStream_t s) {
  if (!evs) return;
  for (int32_t i = from; i < count; ++i)
    if (evs[i]) cudaEventRecord(evs[i], s);
}

}  // namespace

bool signaled_burst_available() { return wait_value32() != nullptr; }

hicache_status signaled_burst(const std::vector<PoolInfo>& pools, const SideSpec& side,
                              const IndexSet& idx, const hicache_opts& o, int32_t layer_begin,
                              int32_t layer_end, cudaStream_t stream, cudaEvent_t* evs) {
  const int32_t count = layer_end - layer_begin;
  // With no row to move no kernel runs, so nothing would ever set the words.
  int64_t rows = 0;
  for (const PoolInfo& pi : pools) rows += pi.page_granular ? idx.n / pi.P : idx.n;
  if (rows == 0) {
    record_from(evs, 0, count, stream);
    return HICACHE_OK;
  }
  WaitValue32Fn wait = wait_value32();
  BurstRes* r = nullptr;
  hicache_status st = wait ? get_res(&r)
                           : fail(HICACHE_ECUDA, "cuStreamWaitValue32 is not available from the driver");
  if (st != HICACHE_OK) {
    record_from(evs, 0, count, stream);
    return st;
  }
  const LaunchCfg cfg{o.max_ctas, o.device_error};
  // The first layer is latency-critical (nothing downstream can start before
  // it), so a large one gets a launch of its own and its event on the caller's
  // stream; the remaining layers share one signalling launch.  A small burst
  // runs as one signalling launch: there a second launch costs more than the
  // first layer gains from the link to itself.
  int64_t layer_bytes = 0;
  for (const PoolInfo& pi : pools)
    layer_bytes += int64_t(pi.T) * moved_row_bytes(pi) * (moves_page_rows(pi) ? idx.n / pi.P : idx.n);
  int32_t first = 0;  // burst-relative index of the first signalled layer
  if (count >= 2 && layer_bytes >= kSplitFirstLayerBytes) {
    st = launch_rows(pools, side, idx.dev_gpu, idx.host_gpu, idx.bits, 0, idx.n, kPagedToDev,
                     layer_begin, layer_begin + 1, cfg, stream);
    cudaError_t e0 = cudaSuccess;
    if (st == HICACHE_OK && evs && evs[0]) e0 = cudaEventRecord(evs[0], stream);
    if (st == HICACHE_OK && e0 != cudaSuccess) st = cuda_fail(e0, "cudaEventRecord(layer_done)");
    if (st != HICACHE_OK) {
      record_from(evs, 0, count, stream);
      return st;
    }
    first = 1;
  }
  const int32_t nsig = count - first;
  // Layers per group: one for layers of kSignalGroupBytes or more, else as
  // many as make up that size, no more than one launch holds.
  int32_t segs_per_layer = 0;
  for (const PoolInfo& pi : pools) segs_per_layer += pi.T;
  const int64_t per_group = std::min<int64_t>(
      {int64_t(nsig), kMaxSegLarge / segs_per_layer,
       std::max<int64_t>(1, (kSignalGroupBytes + layer_bytes - 1) / std::max<int64_t>(1, layer_bytes))});
  uint32_t* words = o.burst_words;
  BurstWords bw{words, words + nsig, words + 2 * int64_t(nsig), words + 3 * int64_t(nsig),
                int32_t(std::max<int64_t>(1, per_group))};
  cudaError_t e = cudaMemsetAsync(words, 0, size_t(kBurstWordsPerLayer) * nsig * sizeof(uint32_t),
                                  stream);
  if (e == cudaSuccess) e = cudaEventRecord(r->fork, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(r->sig, r->fork, 0);
  if (e != cudaSuccess) {
    st = cuda_fail(e, "burst set-up");
    record_from(evs, first, count, stream);
    return st;
  }
  st = launch_rows(pools, side, idx.dev_gpu, idx.host_gpu, idx.bits, 0, idx.n, kPagedToDev,
                   layer_begin + first, layer_end, cfg, stream, &bw);
  if (st != HICACHE_OK) {
    // nothing waits on the words yet: complete the events on the caller's stream
    record_from(evs, first, count, stream);
    return st;
  }
  // one wait per group, on the group's own word, then the group's events
  const int32_t lpg = bw.layers_per_group;
  int32_t i = first;
  while (i < count) {
    const int32_t group = (i - first) / lpg;
    const int32_t last = std::min(count, first + (group + 1) * lpg) - 1;
    const CUresult cr = wait(reinterpret_cast<CUstream>(r->sig),
                             reinterpret_cast<CUdeviceptr>(bw.flag + group), 1u,
                             CU_STREAM_WAIT_VALUE_GEQ);
    if (cr != CUDA_SUCCESS) {
      st = fail(HICACHE_ECUDA, "cuStreamWaitValue32 failed with CUresult " + std::to_string(int(cr)));
      break;
    }
    for (; i <= last; ++i) {
      if (evs && evs[i]) {
        e = cudaEventRecord(evs[i], r->sig);
        if (e != cudaSuccess) {
          st = cuda_fail(e, "cudaEventRecord(layer_done)");
          break;  // evs[i] is recorded on the caller's stream below
        }
      }
    }
    if (st != HICACHE_OK) break;
  }
  // layers whose wait could not be enqueued complete after the launch, on the caller's stream
  record_from(evs, i, count, stream);
  e = cudaEventRecord(r->join, r->sig);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, r->join, 0);
  if (e != cudaSuccess && st == HICACHE_OK) st = cuda_fail(e, "burst join");
  return st;
}

}  // namespace hk
