// row_copy_kernel.cuh -- device code of the row-copy kernel.
//
// Included by zero_copy.cu only.  Kept in a file of its own so that a record of
// hardware counters taken on these kernels can be tied to this exact code.
#pragma once

#include <cuda_runtime.h>

#include "hicache_internal.h"

namespace hk {
namespace {

template <int VEC>
struct VecOf;
template <>
struct VecOf<16> {
  using T = uint4;
};
template <>
struct VecOf<4> {
  using T = uint32_t;
};

template <typename IdxT>
__device__ __forceinline__ int64_t load_index(const void* base, int64_t i) {
  return static_cast<int64_t>(static_cast<const IdxT*>(base)[i]);
}

// Streaming (evict-first) accesses: every byte is touched exactly once.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint32_t* p, const uint32_t& v) { __stcs(p, v); }

// Adds `count` finished tasks to burst group `group`; the warp that completes
// the group publishes its flag.  A group is layers_per_group consecutive layers
// (the last group of the burst may hold fewer).  Called by all 32 lanes of a
// warp.
template <int MAXSEG>
__device__ __forceinline__ void flush_group(const CopyParams<MAXSEG>& p, int group,
                                            uint32_t count, int lane) {
  __threadfence();  // this lane's stores of the group are visible device-wide
  __syncwarp();
  if (lane == 0) {
    const int lpg = p.sig.layers_per_group;
    const int layers = min(lpg, p.sig.burst_layers - group * lpg);
    const uint32_t before = atomicAdd(&p.sig.done[group], count);
    if (int64_t(before) + count == p.sig.tasks_per_layer * layers) {
      __threadfence();
      atomicExch(&p.sig.flag[group], 1u);
    }
  }
}

// Copies the flat chunk range [chunk0, chunk0 + total) of one warp task, where
// chunk c is chunk c % cpr of task row c / cpr.  offs[r] holds the source and
// destination byte offsets of task row r (y < 0 marks a skipped row: a
// destination offset is never negative, a source offset may be); (r, j)
// is the (row, chunk-in-row) position of chunk chunk0 + c0 + lane and advances
// by precomputed quotients, so the loop has no division.  Each lane keeps
// UNROLL chunks in flight.
template <typename V, int VEC, int UNROLL = kUnroll>
__device__ __forceinline__ void copy_chunks(const longlong2* offs, const char* src, char* dst,
                                            const PoolGeom& g, uint32_t chunk0, uint32_t total,
                                            int lane) {
  const uint32_t cpr = g.cpr;
  // advance of 32 * UNROLL chunks as whole rows and a remainder
  const uint32_t qS = UNROLL == kUnroll ? g.qS : uint32_t(32 * UNROLL) / cpr;
  const uint32_t rS = UNROLL == kUnroll ? g.rS : uint32_t(32 * UNROLL) - qS * cpr;
  uint32_t r = (chunk0 + uint32_t(lane)) / cpr;
  uint32_t j = (chunk0 + uint32_t(lane)) - r * cpr;
  for (uint32_t c0 = 0; c0 < total; c0 += 32u * UNROLL) {
    V v[UNROLL];
    int64_t dpos[UNROLL];
    uint32_t rr = r, jj = j;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      dpos[u] = -1;
      if (c0 + uint32_t(lane) + 32u * u < total) {
        const longlong2 o = offs[rr];
        if (o.y >= 0) {
          dpos[u] = o.y + int64_t(jj) * VEC;
          v[u] = ld_stream(reinterpret_cast<const V*>(src + o.x + int64_t(jj) * VEC));
        }
      }
      // advance by 32 chunks
      jj += g.r32;
      rr += g.q32;
      if (jj >= cpr) { jj -= cpr; ++rr; }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (dpos[u] >= 0) st_stream(reinterpret_cast<V*>(dst + dpos[u]), v[u]);
    // advance by 32 * UNROLL chunks
    j += rS;
    r += qS;
    if (j >= cpr) { j -= cpr; ++r; }
  }
}

// Copies the rows of one warp task and returns the task's launch-relative
// segment.  Called by all 32 lanes of a warp; offs is the warp's table of
// kMaxRowsPerTask entries in shared memory.
template <typename IdxT, int MAXSEG, bool LAYER_ROWS, bool DEEP4, bool DEEP>
__device__ __forceinline__ int copy_task(const CopyParams<MAXSEG>& p, int64_t task, int lane,
                                         longlong2* offs) {
  constexpr int kU16 = DEEP ? kUnrollDeep : kUnroll;  // 16-byte chunks in flight per lane
  // segment of this task: last s with seg_task_begin[s] <= task
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seg_task_begin[mid] <= task) lo = mid; else hi = mid - 1;
  }
  const Segment sg = p.seg[lo];
  const PoolGeom& g = p.pool[sg.pool];
  const int64_t t = task - p.seg_task_begin[lo];
  if (LAYER_ROWS && g.layer_rows) {
    // Rows [l0, l0 + nr) of the (token, layer) order of the task's tokens,
    // which start at tok0: row f is layer f % L of token tok0 + f / L, read
    // from that layer's own segment and written next to the token's other
    // layers on the host.  l0 is 0 unless one token spans several tasks.
    const int L = g.num_layers;
    const int64_t tok0 = (t / g.tasks_per_token) * g.tokens_per_task;
    const int l0 = int(t % g.tasks_per_token) * g.rows_per_task;
    const int nr = g.tasks_per_token > 1
                       ? min(g.rows_per_task, L - l0)
                       : int(min(int64_t(g.tokens_per_task), g.nrows - tok0)) * L;
    constexpr int kRowsPerLane = kMaxRowsPerTask / 32;
    int64_t dv[kRowsPerLane], hv[kRowsPerLane];
#pragma unroll
    for (int q = 0; q < kRowsPerLane; ++q) {  // every index load first
      const int r = lane + 32 * q;
      if (r < nr) {
        const int64_t tok = tok0 + (l0 + r) / L;
        dv[q] = load_index<IdxT>(p.dev_idx, p.pair_begin + tok);
        hv[q] = p.paged_idx ? load_index<IdxT>(p.paged_idx, p.pair_begin + tok) : tok;
      }
    }
    bool bad = false;
#pragma unroll
    for (int q = 0; q < kRowsPerLane; ++q) {
      const int r = lane + 32 * q;
      if (r >= nr) break;
      const int f = l0 + r;
      const int l = f - (f / L) * L;
      const int64_t d = dv[q], h = hv[q];
      const bool ok = d >= 0 && d < g.dev_tokens && h >= 0 && h < g.paged_tokens;
      bad = bad || !ok;
      const char* layer_dev = p.seg[lo + l * g.seg_stride].dev;
      const int64_t src = int64_t(reinterpret_cast<uintptr_t>(layer_dev) -
                                  reinterpret_cast<uintptr_t>(sg.dev)) + d * g.row_bytes;
      const int64_t dst = h * g.paged_page_stride + int64_t(l) * g.row_bytes;
      offs[r] = ok ? make_longlong2(src, dst) : make_longlong2(-1, -1);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && p.err) atomicOr(p.err, HICACHE_DEVERR_RANGE);
    __syncwarp();
    const uint32_t total = uint32_t(nr) * g.cpr;
    // 4-byte chunks keep four times as many in flight, so that a lane has as
    // many bytes outstanding on the host link as with 16-byte chunks
    if (g.vec == 16) copy_chunks<uint4, 16, kU16>(offs, sg.dev, sg.paged, g, 0, total, lane);
    else copy_chunks<uint32_t, 4, 4 * kUnroll>(offs, sg.dev, sg.paged, g, 0, total, lane);
    __syncwarp();  // the table is rewritten by the next task
    return lo;
  }
  // A task is rows_per_task whole rows, or one part of a row longer than a task.
  int64_t row0;
  int nr;
  uint32_t chunk0, total;
  if (g.parts_per_row > 1) {
    row0 = t / g.parts_per_row;
    nr = 1;
    chunk0 = uint32_t(t - row0 * g.parts_per_row) * g.part_chunks;
    total = min(g.part_chunks, g.cpr - chunk0);
  } else {
    row0 = t * g.rows_per_task;
    nr = int(min(int64_t(g.rows_per_task), g.nrows - row0));
    chunk0 = 0;
    total = uint32_t(nr) * g.cpr;
  }

  // Each lane resolves rows lane, lane + 32, ... into byte offsets; all index
  // loads are issued before any of them is used.
  constexpr int kRowsPerLane = kMaxRowsPerTask / 32;
  int64_t dv[kRowsPerLane], hv[kRowsPerLane];
#pragma unroll
  for (int q = 0; q < kRowsPerLane; ++q) {
    const int r = lane + 32 * q;
    if (r < nr) {
      const int64_t pair = p.pair_begin + (row0 + r) * g.idx_stride;
      dv[q] = load_index<IdxT>(p.dev_idx, pair);
      hv[q] = p.paged_idx ? load_index<IdxT>(p.paged_idx, pair) : pair - p.pair_begin;
    }
  }
#pragma unroll
  for (int q = 0; q < kRowsPerLane; ++q) {
    const int r = lane + 32 * q;
    if (r >= nr) break;
    const int64_t d = dv[q];
    const int64_t h = hv[q];
    uint32_t e = 0;
    if (d < 0 || d >= g.dev_tokens || h < 0 || h >= g.paged_tokens) {
      e = HICACHE_DEVERR_RANGE;
    } else if (g.idx_div > 1 && ((d % g.idx_div) != 0 || (h % g.idx_div) != 0)) {
      e = HICACHE_DEVERR_PAGE_ALIGN;
    }
    longlong2 o = make_longlong2(-1, -1);
    if (e != 0) {
      if (p.err) atomicOr(p.err, e);
    } else {
      const uint32_t dr = uint32_t(d) / uint32_t(g.idx_div);
      const uint32_t hr = uint32_t(h) / uint32_t(g.idx_div);
      const uint32_t pg = hr / uint32_t(g.rows_per_page);
      const uint32_t t = hr - pg * uint32_t(g.rows_per_page);
      const int64_t doff = int64_t(dr) * g.row_bytes;
      const int64_t poff = int64_t(pg) * g.paged_page_stride + int64_t(t) * g.row_bytes;
      o = p.dir == kDevToPaged ? make_longlong2(doff, poff) : make_longlong2(poff, doff);
    }
    offs[r] = o;
  }
  __syncwarp();
  const char* src = p.dir == kDevToPaged ? sg.dev : sg.paged;
  char* dst = p.dir == kDevToPaged ? sg.paged : sg.dev;
  if (g.vec == 16) copy_chunks<uint4, 16, kU16>(offs, src, dst, g, chunk0, total, lane);
  else copy_chunks<uint32_t, 4, DEEP4 ? 4 * kUnroll : kUnroll>(offs, src, dst, g, chunk0, total, lane);
  __syncwarp();  // the table is rewritten by the next task
  return lo;
}

// LAYER_ROWS: the launch has a pool in the layer-row mode (an all-layer backup
// into a token-major host pool); other launches compile without that branch.
// DEEP4: the launch has a pool that takes 4-byte chunks; they run four times
// as deep, so that a lane keeps as many bytes in flight as with 16-byte
// chunks.  Launches of 16-byte chunks only compile with the shallow loop.
// DEEP: deep tasks (about 4 KiB, kUnrollDeep 16-byte chunks in flight per
// lane) for launches with few CTAs against the host pool.
// WARPS: warps per CTA (kWarpsPerCta, or kWarpsPerCtaWide under a small cap).
template <typename IdxT, int MAXSEG, bool SIGNAL, bool LAYER_ROWS, bool DEEP4, bool DEEP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    row_copy_kernel(const __grid_constant__ CopyParams<MAXSEG> p) {
  __shared__ longlong2 row_offs[WARPS][kMaxRowsPerTask];
  const int lane = threadIdx.x & 31;
  longlong2* offs = row_offs[threadIdx.x >> 5];
  const int64_t ntasks = p.seg_task_begin[p.nseg];
  if constexpr (!SIGNAL) {
    // Static striding: warp w takes tasks w, w + W, w + 2W, ...
    const int64_t warps_total = int64_t(gridDim.x) * WARPS;
    for (int64_t task = int64_t(blockIdx.x) * WARPS + (threadIdx.x >> 5); task < ntasks;
         task += warps_total)
      copy_task<IdxT, MAXSEG, LAYER_ROWS, DEEP4, DEEP>(p, task, lane, offs);
  } else {
    // Tasks are handed out in strict order from one counter, so every task of
    // layer l is taken before any task of layer l+1 and a layer can only wait
    // on the tasks still in flight when its last one was taken.  The next task
    // is claimed before the current one is copied, hiding the atomic's latency.
    uint32_t* next = p.sig.next + p.sig.layer_base;
    const int lpg = p.sig.layers_per_group;
    int cur_group = -1;    // burst group of the tasks counted in `pending`
    uint32_t pending = 0;  // finished tasks of cur_group not yet added to its counter
    uint32_t claim = lane == 0 ? atomicAdd(next, 1u) : 0u;
    int64_t task = __shfl_sync(0xffffffffu, claim, 0);
    while (task < ntasks) {
      claim = lane == 0 ? atomicAdd(next, 1u) : 0u;
      const int layer =
          copy_task<IdxT, MAXSEG, false, DEEP4, DEEP>(p, task, lane, offs) / p.sig.segs_per_layer;
      const int group = (p.sig.layer_base + layer) / lpg;
      if (group != cur_group) {
        if (pending != 0) flush_group(p, cur_group, pending, lane);
        cur_group = group;
        pending = 0;
      }
      ++pending;
      task = __shfl_sync(0xffffffffu, claim, 0);
    }
    if (pending != 0) flush_group(p, cur_group, pending, lane);
    // The last CTA to leave sets every flag of this launch's groups (a launch
    // covers whole groups).  All tasks have been counted by then, so this only
    // guarantees that no waiter can outlive the launch.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t gone = atomicAdd(&p.sig.exits[p.sig.layer_base], 1u);
      if (gone == gridDim.x - 1) {
        __threadfence();
        const int g0 = p.sig.layer_base / lpg;
        const int g1 = (p.sig.layer_base + p.sig.nlayers - 1) / lpg;
        for (int g = g0; g <= g1; ++g) atomicExch(&p.sig.flag[g], 1u);
      }
    }
  }
}

}  // namespace
}  // namespace hk
