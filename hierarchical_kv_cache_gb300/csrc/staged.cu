// staged.cu -- transfers through an HBM staging buffer plus copy-engine DMA.
//
// Prior art: the staged write-back of "[HiCache] Support hybrid-pool staged
// write-back JIT kernel" (sglang PR #28434 summary) packs device rows into a
// page-first staging buffer of a fixed number of pages and then copies it to
// the host.  Here the staging is double-buffered so that the gather of chunk
// k+1 overlaps the link transfer of chunk k, the DMA is one copy per run of
// consecutive host pages (not one per row), and the same idea serves the
// per-layer load in reverse (a 2-D DMA of a group of layer blocks per host
// page, then one scatter launch per chunk of pages; a burst's first layers
// are read zero-copy).  A share of the pages, and pools too small for DMAs of
// their own, move zero-copy on a side stream beside the copy engine.  The
// staged path needs the pairs to be whole host pages in groups of page_size
// (what a page-granular host allocator hands out) and the indices on the
// host, because the DMA spans are planned on the CPU.
#include <cuda_runtime.h>

#include <algorithm>
#include <string>
#include <vector>

#include "burst.h"
#include "staged.h"

namespace hk {

namespace {

hicache_status cuda_fail(cudaError_t e, const std::string& what) {
  return fail(HICACHE_ECUDA, what + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

#define HK_CUDA(call, what)                       \
  do {                                            \
    const cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Events and the internal copy stream, created once per thread and device.
struct StagedRes {
  bool init = false;
  cudaStream_t copy = nullptr;
  cudaStream_t side = nullptr;  // zero-copy share of a staged call
  cudaEvent_t fork = nullptr, join = nullptr, side_done = nullptr, group_start = nullptr;
  cudaEvent_t layer0_done = nullptr, zc_done = nullptr;  // a staged load's zero-copy layers
  cudaEvent_t ready[2] = {nullptr, nullptr};
  cudaEvent_t freed[2] = {nullptr, nullptr};
};

hicache_status get_res(StagedRes** out) {
  static thread_local StagedRes res[64];
  int dev = 0;
  HK_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(HICACHE_EINVAL, "device ordinal above 63");
  StagedRes& r = res[dev];
  if (!r.init) {
    HK_CUDA(cudaStreamCreateWithFlags(&r.copy, cudaStreamNonBlocking), "cudaStreamCreate(copy)");
    HK_CUDA(cudaStreamCreateWithFlags(&r.side, cudaStreamNonBlocking), "cudaStreamCreate(side)");
    cudaEvent_t* evs[10] = {&r.fork,     &r.join,     &r.side_done,   &r.ready[0], &r.ready[1],
                            &r.freed[0], &r.freed[1], &r.group_start, &r.layer0_done, &r.zc_done};
    for (cudaEvent_t* e : evs) HK_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "cudaEventCreate");
    r.init = true;
  }
  *out = &r;
  return HICACHE_OK;
}

// Staging layout: one region per (pool, tensor), each `cap_pages` pages of
// `layers` layer blocks; region offsets are in (pool, tensor) order.
struct StagingLayout {
  int64_t cap_pages = 0;
  std::vector<std::vector<int64_t>> region_off;  // [pool][tensor]
};

StagingLayout layout_for(const std::vector<PoolInfo>& pools, const hicache_opts& o,
                         int32_t layers) {
  StagingLayout s;
  int64_t per_page = 0;
  for (const PoolInfo& pi : pools) per_page += int64_t(pi.T) * layers * pi.P * pi.token_bytes;
  s.cap_pages = per_page > 0 ? int64_t(o.staging_bytes) / per_page : 0;
  int64_t off = 0;
  for (const PoolInfo& pi : pools) {
    std::vector<int64_t> offs;
    const int64_t region = s.cap_pages * layers * pi.P * pi.token_bytes;
    for (int32_t t = 0; t < pi.T; ++t) {
      offs.push_back(off);
      off += region;
    }
    s.region_off.push_back(offs);
  }
  return s;
}

// A staging buffer as a paged side holding `layers` consecutive layers of each
// page, starting at layer `layer_origin`, laid out like a host page of that
// many layers: [page][layer][token][row] for page_first_direct pools,
// [token][layer][row] for page_first pools.
SideSpec staging_side(const std::vector<PoolInfo>& pools, const StagingLayout& lay, char* base,
                      int32_t layers, int32_t layer_origin) {
  SideSpec side;
  side.layer_origin = layer_origin;
  for (size_t p = 0; p < pools.size(); ++p) {
    const PoolInfo& pi = pools[p];
    std::vector<char*> b;
    for (int32_t t = 0; t < pi.T; ++t) b.push_back(base + lay.region_off[p][size_t(t)]);
    const int64_t block = int64_t(pi.P) * pi.token_bytes;  // one (page, layer) block
    if (pi.layout == HICACHE_LAYOUT_PAGE_FIRST_DIRECT) {
      side.layer_stride.push_back(block);
      side.page_stride.push_back(block * layers);
      side.rows_per_page.push_back(moves_page_rows(pi) ? 1 : pi.P);
    } else {
      side.layer_stride.push_back(pi.token_bytes);
      side.page_stride.push_back(int64_t(layers) * pi.token_bytes);
      side.rows_per_page.push_back(1);
    }
    side.paged_tokens.push_back(lay.cap_pages * pi.P);
    side.vec16.push_back(vec16_ok(pi, b, side.layer_stride.back()));
    side.base.push_back(b);
  }
  return side;
}

template <typename T>
int64_t at(const void* p, int64_t i) {
  return int64_t(static_cast<const T*>(p)[i]);
}

hicache_status need_pages(const IndexSet& idx, int32_t P, std::vector<int64_t>* pages) {
  if (!idx.host_cpu)
    return fail(HICACHE_EINVAL, "staged path needs host-located indices (the DMA spans are planned on the CPU)");
  if (!host_page_groups(idx.host_cpu, idx.bits, idx.n, P, pages))
    return fail(HICACHE_EINVAL, "staged path needs the pairs to be whole host pages in groups of page_size");
  return HICACHE_OK;
}

// Entries `which` of a pool list and of a side built over it.
std::vector<PoolInfo> pick(const std::vector<PoolInfo>& pools, const std::vector<size_t>& which) {
  std::vector<PoolInfo> out;
  for (size_t p : which) out.push_back(pools[p]);
  return out;
}

SideSpec pick(const SideSpec& s, const std::vector<size_t>& which) {
  SideSpec out;
  out.layer_origin = s.layer_origin;
  for (size_t p : which) {
    out.vec16.push_back(s.vec16[p]);
    out.base.push_back(s.base[p]);
    out.layer_stride.push_back(s.layer_stride[p]);
    out.page_stride.push_back(s.page_stride[p]);
    out.paged_tokens.push_back(s.paged_tokens[p]);
    out.rows_per_page.push_back(s.rows_per_page[p]);
  }
  return out;
}

// True when the P device slots of every page group are consecutive, so that a
// (page, layer) block is one contiguous span of the device layer buffer.
bool device_pages_consecutive(const void* dev_idx, int32_t bits, int64_t n, int32_t P) {
  for (int64_t k = 0; k < n; k += P) {
    const int64_t d0 = bits == 32 ? at<int32_t>(dev_idx, k) : at<int64_t>(dev_idx, k);
    for (int64_t t = 1; t < P; ++t) {
      const int64_t d = bits == 32 ? at<int32_t>(dev_idx, k + t) : at<int64_t>(dev_idx, k + t);
      if (d != d0 + t) return false;
    }
  }
  return true;
}

// A pool whose host page of all layers (one tensor) is below this many bytes
// moves zero-copy in a staged call that also holds a larger pool: one DMA per
// host page would cost it more in the copy engine's fixed time per copy
// (about 2.4 us device-to-host, 3.3 us host-to-device on GB300) than in
// moving its bytes.  The DSA indexer of a 78-layer model (78 x 64 x 132 B =
// 659 KB per page) is such a pool beside its 5.75 MB latent pages.
constexpr int64_t kDirectPageBytes = int64_t(1) << 20;

// A staged call moves part of its work zero-copy beside the copy engine: the
// copy engine leaves the link idle for its fixed time per copy (2.4-3.3 us on
// GB300) and moves a load's first small layer groups at a fraction of the
// link; SM-issued traffic beside it fills those gaps.
// - A load's first layers, one in kZeroCopyLayerShare.
// - The last pages of a backup, and of each layer group of a load, one in
//   kZeroCopyPageShare.  Against an eighth, a quarter lifted the staged backup
//   from 172 to 175.5 GB/s (Llama-3-8B, 89.0 to 90.9 % of the link), 180 to
//   183 (78-layer) and 173 to 176 (DSv3), and the staged burst from 165 to 174
//   (Llama-3-8B), 169 to 177 (78-layer) and 152 to 161 (DSv3); under a 16-CTA
//   cap beside a GEMM loop both moved as much or more, at a GEMM cost up to 3
//   points higher.
constexpr int64_t kZeroCopyLayerShare = 8;
constexpr int64_t kZeroCopyPageShare = 4;

// Splits a staged call's pools into those that go through staging and the
// small ones that move zero-copy beside them.
void split_pools(const std::vector<PoolInfo>& pools, std::vector<size_t>* staged,
                 std::vector<size_t>* direct) {
  int64_t largest = 0;
  std::vector<int64_t> page(pools.size());
  for (size_t p = 0; p < pools.size(); ++p) {
    page[p] = int64_t(pools[p].L) * pools[p].P * pools[p].token_bytes;
    largest = std::max(largest, page[p]);
  }
  for (size_t p = 0; p < pools.size(); ++p)
    (page[p] < kDirectPageBytes && page[p] < largest ? direct : staged)->push_back(p);
}

// Moves pages [g0, g1) of the pair list for layers [l0, l1) between the device
// slots of `pools` and the staging `side`: whole (page, layer) blocks by bulk
// copy where the pool allows it, rows otherwise.
hicache_status move_staging(const std::vector<PoolInfo>& pools, const SideSpec& side,
                            const IndexSet& idx, bool dev_consecutive, int64_t g0, int64_t g1,
                            Dir dir, int32_t l0, int32_t l1, const LaunchCfg& cfg,
                            cudaStream_t stream) {
  const int32_t P = pools[0].P;
  std::vector<size_t> blocks, rows;
  for (size_t p = 0; p < pools.size(); ++p)
    (dev_consecutive && page_blocks_ok(pools[p], side, p) ? blocks : rows).push_back(p);
  hicache_status st = HICACHE_OK;
  if (!blocks.empty())
    st = launch_page_blocks(pick(pools, blocks), pick(side, blocks), idx.dev_gpu, idx.bits, g0,
                            g1 - g0, dir, l0, l1, cfg, stream);
  if (st == HICACHE_OK && !rows.empty())
    st = launch_rows(pick(pools, rows), pick(side, rows), idx.dev_gpu, nullptr, idx.bits, g0 * P,
                     (g1 - g0) * P, dir, l0, l1, cfg, stream);
  return st;
}

}  // namespace

hicache_status staged_resources_ready() {
  StagedRes* r = nullptr;
  return get_res(&r);
}

bool host_page_groups(const void* host_idx, int32_t bits, int64_t n, int32_t page_size,
                      std::vector<int64_t>* pages) {
  const int64_t P = page_size;
  if (n % P != 0) return false;
  pages->clear();
  pages->reserve(size_t(n / P));
  for (int64_t k = 0; k < n; k += P) {
    const int64_t h0 = bits == 32 ? at<int32_t>(host_idx, k) : at<int64_t>(host_idx, k);
    if (h0 % P != 0) return false;
    for (int64_t t = 1; t < P; ++t) {
      const int64_t h = bits == 32 ? at<int32_t>(host_idx, k + t) : at<int64_t>(host_idx, k + t);
      if (h != h0 + t) return false;
    }
    pages->push_back(h0 / P);
  }
  return true;
}

hicache_status staged_backup(const std::vector<PoolInfo>& all_pools, const hicache_opts& o,
                             const IndexSet& idx, cudaStream_t stream) {
  const int32_t P = all_pools[0].P;
  const int32_t L = all_pools[0].L;
  std::vector<int64_t> hp;
  hicache_status st = need_pages(idx, P, &hp);
  if (st != HICACHE_OK) return st;
  std::vector<size_t> staged_ids, direct_ids;
  split_pools(all_pools, &staged_ids, &direct_ids);
  const std::vector<PoolInfo> pools = pick(all_pools, staged_ids);
  const std::vector<PoolInfo> direct = pick(all_pools, direct_ids);
  const StagingLayout lay = layout_for(pools, o, L);
  if (lay.cap_pages < 1)
    return fail(HICACHE_ENOSTAGE, "staging buffers hold less than one host page of all layers");
  StagedRes* r = nullptr;
  st = get_res(&r);
  if (st != HICACHE_OK) return st;
  cudaStream_t copy = o.copy_stream ? o.copy_stream : r->copy;
  const LaunchCfg cfg{o.max_ctas, o.device_error, /*paged_in_hbm=*/true};
  const LaunchCfg zero_copy{o.max_ctas, o.device_error, /*paged_in_hbm=*/false};
  const int64_t groups = int64_t(hp.size());
  // the last pages move zero-copy beside the copy engine (kZeroCopyPageShare)
  const int64_t zc_pages = groups >= kZeroCopyPageShare
                               ? (groups + kZeroCopyPageShare - 1) / kZeroCopyPageShare
                               : 0;
  const int64_t dma_groups = groups - zc_pages;
  const bool dev_consecutive = device_pages_consecutive(idx.dev_cpu, idx.bits, idx.n, P);
  const SideSpec side[2] = {staging_side(pools, lay, static_cast<char*>(o.staging[0]), L, 0),
                            staging_side(pools, lay, static_cast<char*>(o.staging[1]), L, 0)};
  const bool use_side = zc_pages > 0 || !direct.empty();

  HK_CUDA(cudaEventRecord(r->fork, stream), "cudaEventRecord(fork)");
  HK_CUDA(cudaStreamWaitEvent(copy, r->fork, 0), "cudaStreamWaitEvent(fork)");
  if (use_side) HK_CUDA(cudaStreamWaitEvent(r->side, r->fork, 0), "cudaStreamWaitEvent(fork)");
  // From here on every return joins the copy stream (and the side stream)
  // back into `stream`, also on failure: copies of earlier chunks may still be
  // in flight, and the next call ordered on `stream` may reuse the staging
  // buffers they read.
  auto join = [&](hicache_status s) {
    cudaError_t e = cudaEventRecord(r->join, copy);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, r->join, 0);
    if (e == cudaSuccess && use_side) e = cudaEventRecord(r->side_done, r->side);
    if (e == cudaSuccess && use_side) e = cudaStreamWaitEvent(stream, r->side_done, 0);
    if (e != cudaSuccess && s == HICACHE_OK) s = cuda_fail(e, "staged backup join");
    return s;
  };
  // The zero-copy share on the side stream, concurrent with the gathers and
  // DMAs: every pool's last zc_pages pages and every page of the small pools.
  if (zc_pages > 0) {
    st = launch_rows(pools, host_side(pools), idx.dev_gpu, idx.host_gpu, idx.bits,
                     dma_groups * P, zc_pages * P, kDevToPaged, 0, L, zero_copy, r->side);
    if (st != HICACHE_OK) return join(st);
  }
  if (!direct.empty()) {
    st = launch_rows(direct, host_side(direct), idx.dev_gpu, idx.host_gpu, idx.bits, 0, idx.n,
                     kDevToPaged, 0, L, zero_copy, r->side);
    if (st != HICACHE_OK) return join(st);
  }
#define HK_TRY(call, what)                                  \
  do {                                                      \
    const cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return join(cuda_fail(e_, what)); \
  } while (0)
  for (int64_t k = 0, g0 = 0; g0 < dma_groups; ++k, g0 += lay.cap_pages) {
    const int b = int(k & 1);
    const int64_t g1 = std::min(dma_groups, g0 + lay.cap_pages);
    // the DMA of chunk k-2 must have drained buffer b before the gather reuses it
    if (k >= 2) HK_TRY(cudaStreamWaitEvent(stream, r->freed[b], 0), "cudaStreamWaitEvent(freed)");
    st = move_staging(pools, side[b], idx, dev_consecutive, g0, g1, kDevToPaged, 0, L, cfg, stream);
    if (st != HICACHE_OK) return join(st);
    HK_TRY(cudaEventRecord(r->ready[b], stream), "cudaEventRecord(ready)");
    HK_TRY(cudaStreamWaitEvent(copy, r->ready[b], 0), "cudaStreamWaitEvent(ready)");
    for (size_t p = 0; p < pools.size(); ++p) {
      const PoolInfo& pi = pools[p];
      const int64_t page_bytes = int64_t(L) * pi.P * pi.token_bytes;  // one host page, all layers
      for (int32_t t = 0; t < pi.T; ++t) {
        for (int64_t j = g0; j < g1;) {
          int64_t e = j + 1;
          while (e < g1 && hp[size_t(e)] == hp[size_t(e - 1)] + 1) ++e;
          char* dst = pi.host[size_t(t)] + hp[size_t(j)] * page_bytes;
          const char* src = side[b].base[p][size_t(t)] + (j - g0) * page_bytes;
          HK_TRY(cudaMemcpyAsync(dst, src, size_t((e - j) * page_bytes), cudaMemcpyDeviceToHost, copy),
                 "cudaMemcpyAsync(staging -> host)");
          j = e;
        }
      }
    }
    HK_TRY(cudaEventRecord(r->freed[b], copy), "cudaEventRecord(freed)");
  }
#undef HK_TRY
  return join(HICACHE_OK);
}

// The copy engine costs about 3 microseconds per copy on GB300, whatever the
// number of streams or host threads issuing them: a 128 KiB copy (one layer of
// one 64-token page of 2 KiB rows) moves 33 GB/s, a 512 KiB copy 106 GB/s,
// 2 MiB 170 GB/s and 4 MiB 186 GB/s (host to device).  The staged load
// therefore copies a group of consecutive layers of each host page per DMA
// (they are adjacent in a page-first host page).  After the zero-copy first
// layers the groups grow fourfold, 4, 16, ... layers, until one copy carries
// about this many bytes; a tail shorter than its group is merged or split
// evenly.  A 32-layer burst of 128 KiB blocks runs as 4 zero-copy layers, then
// groups of 4 and 24; a 78-layer burst of 72 KiB blocks as 10 zero-copy
// layers, then 4, 16 and 48.
constexpr int64_t kDmaCopyTargetBytes = int64_t(4) << 20;
constexpr int32_t kGroupGrowth = 4;
// A group too large for the staging to hold every page at once moves in
// chunks of pages; a chunk holds at least this many pages (or all of them),
// so that the per-chunk scatter launch and stream hand-offs stay small next
// to its copies.
constexpr int64_t kMinChunkPages = 32;

hicache_status staged_load(const std::vector<PoolInfo>& all_pools, const hicache_opts& o,
                           const IndexSet& idx, int32_t layer_begin, int32_t layer_end,
                           cudaStream_t stream, cudaEvent_t* layer_done) {
  const int32_t P = all_pools[0].P;
  const int32_t L = all_pools[0].L;
  const int32_t count = layer_end - layer_begin;
  int32_t recorded = 0;  // layer events recorded so far, in order
  cudaStream_t forked = nullptr;  // the copy stream once it has forked from `stream`
  bool side_used = false;         // the side stream holds zero-copy page shares
  StagedRes* r = nullptr;
  auto finish = [&](hicache_status s) {
    // A failed load joins the copy stream back into `stream` (copies into the
    // staging buffers may still be in flight), and the side stream, and then
    // completes every remaining layer event.
    cudaError_t e = cudaSuccess;
    if (forked) {
      e = cudaEventRecord(r->join, forked);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, r->join, 0);
    }
    if (e == cudaSuccess && side_used) e = cudaEventRecord(r->side_done, r->side);
    if (e == cudaSuccess && side_used) e = cudaStreamWaitEvent(stream, r->side_done, 0);
    if (e != cudaSuccess && s == HICACHE_OK) s = cuda_fail(e, "staged load join");
    for (int32_t i = recorded; i < count; ++i)
      if (layer_done && layer_done[i]) cudaEventRecord(layer_done[i], stream);
    return s;
  };
  std::vector<int64_t> hp;
  hicache_status st = need_pages(idx, P, &hp);
  if (st != HICACHE_OK) return finish(st);
  std::vector<size_t> staged_ids, direct_ids;
  split_pools(all_pools, &staged_ids, &direct_ids);
  const std::vector<PoolInfo> pools = pick(all_pools, staged_ids);
  const std::vector<PoolInfo> direct = pick(all_pools, direct_ids);
  const SideSpec direct_side = host_side(direct);
  if (layout_for(pools, o, 1).cap_pages < 1)
    return finish(fail(HICACHE_ENOSTAGE, "staging buffers hold less than one host page of one layer"));
  st = get_res(&r);
  if (st != HICACHE_OK) return finish(st);
  cudaStream_t copy = o.copy_stream ? o.copy_stream : r->copy;
  const LaunchCfg cfg{o.max_ctas, o.device_error, /*paged_in_hbm=*/true};
  const LaunchCfg zero_copy{o.max_ctas, o.device_error, /*paged_in_hbm=*/false};
  const int64_t groups = int64_t(hp.size());
  if (groups == 0) return finish(HICACHE_OK);  // nothing to move; the events still fire
  // The last pages of every layer group (kZeroCopyPageShare) are read
  // zero-copy on the side stream while the copy engine moves the group's
  // other pages.
  const int64_t zc_pages = groups >= kZeroCopyPageShare
                               ? (groups + kZeroCopyPageShare - 1) / kZeroCopyPageShare
                               : 0;
  const int64_t dma_groups = groups - zc_pages;
  const bool group_side = zc_pages > 0 || !direct.empty();  // a group has side-stream work
  const bool dev_consecutive = device_pages_consecutive(idx.dev_cpu, idx.bits, idx.n, P);
  int64_t max_block = 1;
  for (const PoolInfo& pi : pools) max_block = std::max(max_block, int64_t(pi.P) * pi.token_bytes);
  const int32_t g_cap = int32_t(std::min<int64_t>(
      count, std::max<int64_t>(1, (kDmaCopyTargetBytes + max_block - 1) / max_block)));

#define HK_TRY(call, what)                                    \
  do {                                                        \
    const cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return finish(cuda_fail(e_, what)); \
  } while (0)

  // The first layers of a burst of two or more (one in kZeroCopyLayerShare, at
  // least one) are read zero-copy: the SMs read the host pool directly, one
  // launch and event per layer.  Through the copy engine the first layer
  // would cost one small copy per host page before its event, and the first
  // layer groups would move in copies too small for the link.  The copy stream
  // forks once the first layer's launch is enqueued, so that layer has the
  // link to itself; the other zero-copy layers share it with the copy
  // engine's first, smaller groups, whose copies leave the link idle for part
  // of their time.
  const int32_t zc_layers =
      count >= 2 ? int32_t(std::max<int64_t>(1, (count + kZeroCopyLayerShare - 1) / kZeroCopyLayerShare))
                 : 0;
  // The zero-copy layers run on the side stream, so that the scatters of the
  // first layer groups (on `stream`) do not queue behind them and the copy
  // engine's staging buffers keep turning over.  Their events are recorded
  // on that stream; the first group's events wait for them, so the events
  // still complete in layer order.
  auto load_direct_layer = [&](int32_t k) {
    const hicache_status s = launch_rows(all_pools, host_side(all_pools), idx.dev_gpu,
                                         idx.host_gpu, idx.bits, 0, idx.n, kPagedToDev, k, k + 1,
                                         zero_copy, r->side);
    if (s != HICACHE_OK) return s;
    if (layer_done && layer_done[k - layer_begin]) {
      const cudaError_t e = cudaEventRecord(layer_done[k - layer_begin], r->side);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(layer_done)");
    }
    ++recorded;
    return HICACHE_OK;
  };
  HK_TRY(cudaEventRecord(r->fork, stream), "cudaEventRecord(fork)");
  if (zc_layers > 0) {
    HK_TRY(cudaStreamWaitEvent(r->side, r->fork, 0), "cudaStreamWaitEvent(fork)");
    side_used = true;
    st = load_direct_layer(layer_begin);
    if (st != HICACHE_OK) return finish(st);
    // the copy engine starts once layer 0 has landed: layer 0 has the link to itself
    HK_TRY(cudaEventRecord(r->layer0_done, r->side), "cudaEventRecord(layer 0 done)");
    HK_TRY(cudaStreamWaitEvent(copy, r->layer0_done, 0), "cudaStreamWaitEvent(layer 0 done)");
  } else {
    HK_TRY(cudaStreamWaitEvent(copy, r->fork, 0), "cudaStreamWaitEvent(fork)");
  }
  forked = copy;
  if (zc_layers >= 3 && o.burst_words && signaled_burst_available()) {
    // the other zero-copy layers as one signalling launch (fewer launches to
    // wait for SMs when a concurrent kernel holds them); it records their
    // events on every return path
    st = signaled_burst(all_pools, host_side(all_pools), idx, o, layer_begin + 1,
                        layer_begin + zc_layers, r->side, layer_done ? layer_done + 1 : nullptr);
    recorded += zc_layers - 1;
    if (st != HICACHE_OK) return finish(st);
  } else {
    for (int32_t k = layer_begin + 1; k < layer_begin + zc_layers; ++k) {
      st = load_direct_layer(k);
      if (st != HICACHE_OK) return finish(st);
    }
  }
  if (zc_layers > 0) HK_TRY(cudaEventRecord(r->zc_done, r->side), "cudaEventRecord(zero-copy layers done)");
  bool first_group = true;
  const int32_t first = layer_begin + zc_layers;
  int64_t step = 0;
  // the groups start small whatever the zero-copy share, so that the layer
  // events keep arriving in steps (a consumer starts on them early)
  int32_t g_want = first == layer_begin ? 1 : std::min(g_cap, kGroupGrowth);
  for (int32_t l = first, g = 1; l < layer_end; l += g) {
    // the next group size; a tail shorter than the group joins it (or, when
    // both would not fit in one copy, the rest is split in two even groups)
    const int32_t remaining = layer_end - l;
    g = std::min(g_want, remaining);
    if (remaining > g && remaining - g < g) g = remaining <= g_cap ? remaining : (remaining + 1) / 2;
    // the largest such group whose chunks hold kMinChunkPages pages, or every
    // page; one layer per group when not even that fits
    while (g > 1 && layout_for(pools, o, g).cap_pages < std::min(dma_groups, kMinChunkPages)) --g;
    g_want = std::min(g_cap, kGroupGrowth * g_want);
    const StagingLayout lay = layout_for(pools, o, g);
    for (int64_t g0 = 0; g0 < dma_groups; g0 += lay.cap_pages, ++step) {
      const int b = int(step & 1);
      const int64_t g1 = std::min(dma_groups, g0 + lay.cap_pages);
      const bool last_chunk = g1 == dma_groups;
      const SideSpec side = staging_side(pools, lay, static_cast<char*>(o.staging[b]), g, l);
      // the scatter of step-2 must have read buffer b before the DMA refills it
      if (step >= 2) HK_TRY(cudaStreamWaitEvent(copy, r->freed[b], 0), "cudaStreamWaitEvent(freed)");
      if (g0 == 0 && group_side) {
        // The group's zero-copy work starts with its first copies, on the side
        // stream: the staged pools' last pages, and every page of the small
        // pools.  One launch each per group keeps the launch count low, which
        // matters when a concurrent kernel holds the SMs.
        HK_TRY(cudaEventRecord(r->group_start, copy), "cudaEventRecord(group start)");
        HK_TRY(cudaStreamWaitEvent(r->side, r->group_start, 0), "cudaStreamWaitEvent(group start)");
        side_used = true;
        if (zc_pages > 0) {
          st = launch_rows(pools, host_side(pools), idx.dev_gpu, idx.host_gpu, idx.bits,
                           dma_groups * P, zc_pages * P, kPagedToDev, l, l + g, zero_copy, r->side);
          if (st != HICACHE_OK) return finish(st);
        }
        if (!direct.empty()) {
          st = launch_rows(direct, direct_side, idx.dev_gpu, idx.host_gpu, idx.bits, 0, idx.n,
                           kPagedToDev, l, l + g, zero_copy, r->side);
          if (st != HICACHE_OK) return finish(st);
        }
        HK_TRY(cudaEventRecord(r->side_done, r->side), "cudaEventRecord(side done)");
      }
      for (size_t p = 0; p < pools.size(); ++p) {
        const PoolInfo& pi = pools[p];
        const int64_t R = pi.token_bytes;
        const int64_t block = int64_t(pi.P) * R;  // one (page, layer) block
        const int64_t host_page = block * L;
        const bool direct_layout = pi.layout == HICACHE_LAYOUT_PAGE_FIRST_DIRECT;
        for (int32_t t = 0; t < pi.T; ++t) {
          for (int64_t j = g0; j < g1;) {
            int64_t e = j + 1;
            while (e < g1 && hp[size_t(e)] == hp[size_t(e - 1)] + 1) ++e;
            char* dst = side.base[p][size_t(t)] + (j - g0) * block * g;
            const char* page0 = pi.host[size_t(t)] + hp[size_t(j)] * host_page;
            // direct: layers l..l+g-1 of a page are one contiguous span, pages
            // host_page apart; page_first: they are contiguous per token, tokens
            // L * R apart
            const cudaError_t ce =
                direct_layout
                    ? cudaMemcpy2DAsync(dst, size_t(block * g), page0 + int64_t(l) * block,
                                        size_t(host_page), size_t(block * g), size_t(e - j),
                                        cudaMemcpyHostToDevice, copy)
                    : cudaMemcpy2DAsync(dst, size_t(R * g), page0 + int64_t(l) * R,
                                        size_t(L) * size_t(R), size_t(R * g),
                                        size_t((e - j) * pi.P), cudaMemcpyHostToDevice, copy);
            HK_TRY(ce, "cudaMemcpy2DAsync(host -> staging)");
            j = e;
          }
        }
      }
      HK_TRY(cudaEventRecord(r->ready[b], copy), "cudaEventRecord(ready)");
      HK_TRY(cudaStreamWaitEvent(stream, r->ready[b], 0), "cudaStreamWaitEvent(ready)");
      // one scatter launch per chunk, all of the group's layers
      st = move_staging(pools, side, idx, dev_consecutive, g0, g1, kPagedToDev, l, l + g, cfg,
                        stream);
      if (st != HICACHE_OK) return finish(st);
      if (last_chunk) {
        // the group has landed once its zero-copy work has too: its events
        // (the first group's also come after the zero-copy layers')
        if (group_side)
          HK_TRY(cudaStreamWaitEvent(stream, r->side_done, 0), "cudaStreamWaitEvent(side done)");
        else if (first_group && zc_layers > 0)
          HK_TRY(cudaStreamWaitEvent(stream, r->zc_done, 0), "cudaStreamWaitEvent(zero-copy layers)");
        first_group = false;
        for (int32_t k = l; k < l + g; ++k) {
          if (layer_done && layer_done[k - layer_begin])
            HK_TRY(cudaEventRecord(layer_done[k - layer_begin], stream), "cudaEventRecord(layer_done)");
          ++recorded;
        }
      }
      HK_TRY(cudaEventRecord(r->freed[b], stream), "cudaEventRecord(freed)");
    }
  }
  // the side stream's work joins `stream` before the call returns
  if (side_used) {
    HK_TRY(cudaEventRecord(r->side_done, r->side), "cudaEventRecord(side done)");
    HK_TRY(cudaStreamWaitEvent(stream, r->side_done, 0), "cudaStreamWaitEvent(side done)");
  }
#undef HK_TRY
  return HICACHE_OK;
}

hicache_path choose_path(const std::vector<PoolInfo>& pools, const hicache_opts& o,
                         const IndexSet& idx, Dir dir, int32_t layers) {
  // Measured on GB300 (NVLink-C2C host link): with the SMs to itself the
  // zero-copy kernel reaches the copy-engine bandwidth and was at least as
  // fast as the staged path at every point of the row size / page size /
  // length sweep.  Its bandwidth grows with its CTAs, though, until about 16
  // (of 16 warps) fill the link, while the staged path needs SMs only for
  // short gather and scatter kernels.  So when the caller caps the copy's
  // CTAs to keep the SMs for compute, below the crossover (5 CTAs beside a
  // bf16 GEMM loop) the staged path is faster, where it may run and its DMAs
  // are large.
  const int32_t below = dir == kDevToPaged ? HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP
                                           : HICACHE_AUTO_STAGED_BELOW_CTAS_LOAD;
  if (o.max_ctas <= 0 || o.max_ctas >= below) return HICACHE_PATH_ZERO_COPY;
  if (dir == kPagedToDev && layers < 2) return HICACHE_PATH_ZERO_COPY;
  if (!o.staging[0] || !o.staging[1] || o.staging_bytes == 0) return HICACHE_PATH_ZERO_COPY;
  if (o.index_location != HICACHE_INDEX_HOST || !idx.host_cpu || idx.n == 0)
    return HICACHE_PATH_ZERO_COPY;
  int64_t largest = 0;
  for (const PoolInfo& pi : pools)
    largest = std::max(largest, int64_t(pi.L) * pi.P * pi.token_bytes);
  if (largest < kDirectPageBytes) return HICACHE_PATH_ZERO_COPY;
  std::vector<int64_t> hp;
  if (!host_page_groups(idx.host_cpu, idx.bits, idx.n, pools[0].P, &hp))
    return HICACHE_PATH_ZERO_COPY;
  std::vector<size_t> staged_ids, direct_ids;
  split_pools(pools, &staged_ids, &direct_ids);
  const int32_t staged_layers = dir == kDevToPaged ? pools[0].L : 1;
  if (layout_for(pick(pools, staged_ids), o, staged_layers).cap_pages < 1)
    return HICACHE_PATH_ZERO_COPY;
  return HICACHE_PATH_STAGED;
}

}  // namespace hk
