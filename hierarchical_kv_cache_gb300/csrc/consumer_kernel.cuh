// consumer_kernel.cuh -- device code of the synthetic consumer (checksum) kernel.
//
// Included by zero_copy.cu only.  It stands in for the attention layer that
// waits on a layer-done event: it reads every loaded row of one layer.
#pragma once

#include <cuda_runtime.h>

#include "hicache_internal.h"

namespace hk {
namespace {

// Synthetic consumer: sum of the 32-bit words of the rows at the given slots.
// One warp per row at a time; lanes read 16-byte chunks (4-byte words for a
// row or base that is not 16-aligned), several chunks in flight per lane.
template <typename IdxT>
__global__ void __launch_bounds__(kThreadsPerCta)
    checksum_kernel(const char* layer, int64_t row_bytes, const IdxT* idx, int64_t n,
                    int64_t dev_slots, unsigned long long* out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = int64_t(gridDim.x) * kWarpsPerCta;
  const bool vec16 = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(layer) % 16 == 0;
  unsigned long long acc = 0;
  for (int64_t i = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); i < n;
       i += warps_total) {
    const int64_t d = static_cast<int64_t>(idx[i]);
    if (d < 0 || d >= dev_slots) continue;
    const char* row = layer + d * row_bytes;
    if (vec16) {
      const uint4* v = reinterpret_cast<const uint4*>(row);
      const int64_t chunks = row_bytes / 16;
#pragma unroll 4
      for (int64_t k = lane; k < chunks; k += 32) {
        const uint4 x = __ldcs(v + k);
        acc += uint64_t(x.x) + x.y + x.z + x.w;
      }
    } else {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(row);
      for (int64_t k = lane; k < row_bytes / 4; k += 32) acc += w[k];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if (lane == 0 && acc != 0) atomicAdd(out, acc);
}

}  // namespace
}  // namespace hk
