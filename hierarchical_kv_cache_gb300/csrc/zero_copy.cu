// zero_copy.cu -- the row-gather copy kernel and its launcher.
//
// One kernel moves rows between layer-first device buffers and a page-first
// "paged" side.  The paged side is either the pinned host pool itself, read or
// written by the SMs through its mapping (zero-copy path: all-layer backup and
// per-layer load-back of "[HiCache] Support hybrid-pool staged write-back JIT
// kernel" and "[HiCache] Run the host->device load-back enqueue on a loader
// thread"), or an HBM staging buffer with the same page-first structure (staged
// path).
//
// Work decomposition: a warp task is up to 32 rows of one segment (one pool,
// tensor and layer).  Lane r loads pair r of the task, checks it and turns it
// into a source and a destination byte offset.  The task's rows are then
// treated as one flat array of VEC-byte chunks: lane k of an iteration copies
// chunk c0 + k, fetching the offsets of that chunk's row from the owning lane
// with a shuffle.  Rows that are adjacent on both sides therefore produce
// fully coalesced 512-byte warp accesses whatever the row size, which is how
// contiguous index runs are merged without any run table.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

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

template <typename IdxT, int VEC, int MAXSEG>
__global__ void __launch_bounds__(kThreadsPerCta)
    row_copy_kernel(const __grid_constant__ CopyParams<MAXSEG> p) {
  using V = typename VecOf<VEC>::T;
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = int64_t(gridDim.x) * kWarpsPerCta;
  const int64_t ntasks = p.seg_task_begin[p.nseg];
  for (int64_t task = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); task < ntasks;
       task += warps_total) {
    // segment of this task: last s with seg_task_begin[s] <= task
    int lo = 0, hi = p.nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.seg_task_begin[mid] <= task) lo = mid; else hi = mid - 1;
    }
    const Segment sg = p.seg[lo];
    const PoolGeom& g = p.pool[sg.pool];
    const int64_t row0 = (task - p.seg_task_begin[lo]) * g.rows_per_task;
    const int nr = int(min(int64_t(g.rows_per_task), g.nrows - row0));

    // Lane r < nr resolves row row0 + r into byte offsets (-1 marks a skipped row).
    int64_t src_off = -1, dst_off = -1;
    if (lane < nr) {
      const int64_t pair = p.pair_begin + (row0 + lane) * g.idx_stride;
      const int64_t d = load_index<IdxT>(p.dev_idx, pair);
      const int64_t h = p.paged_idx ? load_index<IdxT>(p.paged_idx, pair) : pair - p.pair_begin;
      uint32_t e = 0;
      if (d < 0 || d >= g.dev_tokens || h < 0 || h >= g.paged_tokens) {
        e = HICACHE_DEVERR_RANGE;
      } else if (g.idx_div > 1 && ((d % g.idx_div) != 0 || (h % g.idx_div) != 0)) {
        e = HICACHE_DEVERR_PAGE_ALIGN;
      }
      if (e != 0) {
        if (p.err) atomicOr(p.err, e);
      } else {
        const uint32_t dr = uint32_t(d) / uint32_t(g.idx_div);
        const uint32_t hr = uint32_t(h) / uint32_t(g.idx_div);
        const uint32_t pg = hr / uint32_t(g.rows_per_page);
        const uint32_t t = hr - pg * uint32_t(g.rows_per_page);
        const int64_t doff = int64_t(dr) * g.row_bytes;
        const int64_t poff = int64_t(pg) * g.paged_page_stride + int64_t(t) * g.row_bytes;
        src_off = p.dir == kDevToPaged ? doff : poff;
        dst_off = p.dir == kDevToPaged ? poff : doff;
      }
    }
    const char* src = p.dir == kDevToPaged ? sg.dev : sg.paged;
    char* dst = p.dir == kDevToPaged ? sg.paged : sg.dev;

    // Flat chunk loop.  (r, j) = (row, chunk-in-row) of chunk c0 + lane.
    const uint32_t cpr = g.cpr;
    const uint32_t total = uint32_t(nr) * cpr;
    uint32_t r = uint32_t(lane) / cpr;
    uint32_t j = uint32_t(lane) - r * cpr;
    for (uint32_t c0 = 0; c0 < total; c0 += 32u * kUnroll) {
      V v[kUnroll];
      int64_t dpos[kUnroll];
      uint32_t rr = r, jj = j;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = c0 + uint32_t(lane) + 32u * u;
        const int owner = int(min(rr, 31u));
        const int64_t so = __shfl_sync(0xffffffffu, src_off, owner);
        const int64_t dof = __shfl_sync(0xffffffffu, dst_off, owner);
        const bool live = c < total && so >= 0;
        dpos[u] = live ? dof + int64_t(jj) * VEC : -1;
        if (live) v[u] = ld_stream(reinterpret_cast<const V*>(src + so + int64_t(jj) * VEC));
        // advance by 32 chunks
        jj += g.r32;
        rr += g.q32;
        if (jj >= cpr) { jj -= cpr; ++rr; }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (dpos[u] >= 0) st_stream(reinterpret_cast<V*>(dst + dpos[u]), v[u]);
      // advance by 32 * kUnroll chunks
      j += g.rS;
      r += g.qS;
      if (j >= cpr) { j -= cpr; ++r; }
    }
  }
}

// Synthetic consumer: sum of the 32-bit words of the rows at the given slots.
template <typename IdxT>
__global__ void __launch_bounds__(kThreadsPerCta)
    checksum_kernel(const char* layer, int64_t row_bytes, const IdxT* idx, int64_t n,
                    int64_t dev_slots, unsigned long long* out) {
  unsigned long long acc = 0;
  const int64_t words = row_bytes / 4;
  for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int64_t d = static_cast<int64_t>(idx[i]);
    if (d < 0 || d >= dev_slots) continue;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(layer + d * row_bytes);
    for (int64_t k = threadIdx.x; k < words; k += blockDim.x) acc += w[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicAdd(out, acc);
}

hicache_status cuda_fail(cudaError_t e, const char* what) {
  return fail(HICACHE_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                 cudaGetErrorString(e) + ")");
}

template <int MAXSEG>
hicache_status launch_segments(const CopyParams<MAXSEG>& prm, int32_t index_bits, bool vec16,
                               int64_t ntasks, const LaunchCfg& cfg, cudaStream_t stream) {
  if (ntasks <= 0) return HICACHE_OK;
  int max_ctas = cfg.max_ctas > 0 ? cfg.max_ctas : device_sm_count() * kDefaultCtasPerSm;
  const int64_t want = (ntasks + kWarpsPerCta - 1) / kWarpsPerCta;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, max_ctas)));
  if (index_bits == 32) {
    if (vec16) row_copy_kernel<int32_t, 16, MAXSEG><<<grid, kThreadsPerCta, 0, stream>>>(prm);
    else row_copy_kernel<int32_t, 4, MAXSEG><<<grid, kThreadsPerCta, 0, stream>>>(prm);
  } else {
    if (vec16) row_copy_kernel<int64_t, 16, MAXSEG><<<grid, kThreadsPerCta, 0, stream>>>(prm);
    else row_copy_kernel<int64_t, 4, MAXSEG><<<grid, kThreadsPerCta, 0, stream>>>(prm);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "row copy kernel launch");
  count_launch();
  return HICACHE_OK;
}

}  // namespace

namespace {
std::atomic<int64_t> g_launches{0};
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
int64_t kernel_launches() { return g_launches.load(std::memory_order_relaxed); }

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      sms = 152;
    cache[dev] = sms;
  }
  return cache[dev];
}

int64_t moved_row_bytes(const PoolInfo& pi) {
  return pi.page_granular ? pi.token_bytes * pi.P : pi.token_bytes;
}

bool vec16_ok(const std::vector<PoolInfo>& pools) {
  for (const PoolInfo& pi : pools) {
    if (moved_row_bytes(pi) % 16 != 0) return false;
    for (char* ptr : pi.dev)
      if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    for (char* ptr : pi.host)
      if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
  }
  return true;
}

void fill_geometry(const PoolInfo& pi, int64_t npairs, int vec, int64_t paged_page_stride,
                   int64_t paged_tokens, PoolGeom* g) {
  const int64_t R = moved_row_bytes(pi);
  g->row_bytes = R;
  g->paged_page_stride = paged_page_stride;
  g->dev_tokens = pi.device_slots;
  g->paged_tokens = paged_tokens;
  g->rows_per_page = pi.page_granular ? 1 : pi.P;
  g->idx_stride = pi.page_granular ? pi.P : 1;
  g->idx_div = pi.page_granular ? pi.P : 1;
  g->nrows = pi.page_granular ? npairs / pi.P : npairs;
  g->cpr = uint32_t(R / vec);
  g->q32 = 32u / g->cpr;
  g->r32 = 32u % g->cpr;
  g->qS = uint32_t(32 * kUnroll) / g->cpr;
  g->rS = uint32_t(32 * kUnroll) % g->cpr;
  const int64_t rpt = (int64_t(32) * kUnroll + g->cpr - 1) / g->cpr;
  g->rows_per_task = int32_t(std::min<int64_t>(32, std::max<int64_t>(1, rpt)));
  g->tasks_per_seg = (g->nrows + g->rows_per_task - 1) / g->rows_per_task;
}

hicache_status launch_rows(const std::vector<PoolInfo>& pools, const SideSpec& side,
                           const void* dev_idx, const void* paged_idx, int32_t index_bits,
                           int64_t pair_begin, int64_t npairs, Dir dir, int32_t layer_begin,
                           int32_t layer_end, const LaunchCfg& cfg, cudaStream_t stream) {
  if (npairs <= 0 || layer_end <= layer_begin) return HICACHE_OK;
  const bool vec16 = side.vec16;
  const int vec = vec16 ? 16 : 4;
  const bool small = int64_t(layer_end - layer_begin) * int64_t(pools.size()) * 2 <= kMaxSegSmall;

  auto run = [&](auto& prm, int maxseg) -> hicache_status {
    prm.dev_idx = dev_idx;
    prm.paged_idx = paged_idx;
    prm.err = cfg.err;
    prm.dir = dir;
    prm.pair_begin = pair_begin;
    for (size_t p = 0; p < pools.size(); ++p)
      fill_geometry(pools[p], npairs, vec, side.page_stride[p], side.paged_tokens[p], &prm.pool[p]);
    int nseg = 0;
    int64_t tasks = 0;
    for (int32_t l = layer_begin; l < layer_end; ++l) {
      for (size_t p = 0; p < pools.size(); ++p) {
        const PoolInfo& pi = pools[p];
        for (int32_t t = 0; t < pi.T; ++t) {
          Segment& s = prm.seg[nseg];
          s.dev = pi.dev[size_t(t) * pi.L + l];
          s.paged = side.base[p][size_t(t)] + int64_t(l - side.layer_origin) * side.layer_stride[p];
          s.pool = int32_t(p);
          s.pad = 0;
          prm.seg_task_begin[nseg] = tasks;
          tasks += prm.pool[p].tasks_per_seg;
          ++nseg;
          if (nseg == maxseg) {
            prm.nseg = nseg;
            prm.seg_task_begin[nseg] = tasks;
            const hicache_status st = launch_segments(prm, index_bits, vec16, tasks, cfg, stream);
            if (st != HICACHE_OK) return st;
            nseg = 0;
            tasks = 0;
          }
        }
      }
    }
    if (nseg > 0) {
      prm.nseg = nseg;
      prm.seg_task_begin[nseg] = tasks;
      return launch_segments(prm, index_bits, vec16, tasks, cfg, stream);
    }
    return HICACHE_OK;
  };
  if (small) {
    CopyParams<kMaxSegSmall> prm{};
    return run(prm, kMaxSegSmall);
  }
  static thread_local CopyParams<kMaxSegLarge> prm_large;
  prm_large = CopyParams<kMaxSegLarge>{};
  return run(prm_large, kMaxSegLarge);
}

hicache_status launch_checksum(const PoolInfo& pool, int32_t tensor, int32_t layer,
                               const void* dev_idx, int32_t index_bits, int64_t n, uint64_t* out,
                               cudaStream_t stream) {
  if (n <= 0) return HICACHE_OK;
  const char* base = pool.dev[size_t(tensor) * pool.L + layer];
  const int grid = int(std::min<int64_t>(n, int64_t(device_sm_count()) * 4));
  auto* o = reinterpret_cast<unsigned long long*>(out);
  if (index_bits == 32)
    checksum_kernel<int32_t><<<grid, kThreadsPerCta, 0, stream>>>(
        base, pool.token_bytes, static_cast<const int32_t*>(dev_idx), n, pool.device_slots, o);
  else
    checksum_kernel<int64_t><<<grid, kThreadsPerCta, 0, stream>>>(
        base, pool.token_bytes, static_cast<const int64_t*>(dev_idx), n, pool.device_slots, o);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "checksum kernel launch");
  count_launch();
  return HICACHE_OK;
}

}  // namespace hk
