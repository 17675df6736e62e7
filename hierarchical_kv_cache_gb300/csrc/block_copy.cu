// block_copy.cu -- whole (page, layer) blocks between the device pool and HBM
// staging, moved by the SM's bulk-copy (TMA) engine.
//
// The staged path of "[HiCache] Support hybrid-pool staged write-back JIT
// kernel" (sglang PR #28434 summary) packs device rows into a page-first
// staging buffer before the link transfer, and the staged load unpacks them.
// When a page's P device slots are consecutive and the pool's host layout is
// page_first_direct, one (page, layer) block is P * R contiguous bytes on both
// sides, so the copy needs no per-row work at all: it is a list of equal
// blocks.  One thread of each CTA streams 16 KiB chunks of its
// blocks global -> shared -> global with cp.async.bulk: a load lands in a
// shared-memory stage and completes a transaction count on that stage's
// mbarrier, the thread then issues the bulk store of the stage and reuses it
// once the store has read it.  Four stages keep three loads in flight per CTA,
// and three CTAs share an SM, so about 150 KiB per SM are in flight: enough to
// cover HBM latency, with no register or issue pressure.
//
// The 32 lanes of the CTA resolve the addresses of 32 chunks at a time (one
// index load each, all in flight together), so the issuing thread never
// waits on an index load.
//
// Every wait is bounded: a stage that has not landed within one second of
// %globaltimer sets HICACHE_DEVERR_TIMEOUT, waits (again bounded) for the
// CTA's loads still in flight and for its stores, and the CTA returns.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <type_traits>

#include "hicache_internal.h"

namespace hk {

namespace {

constexpr int kStages = 4;
constexpr uint32_t kChunk = 16384;         // bytes per bulk copy
constexpr int kBlockCtasPerSm = 3;         // 64 KiB of shared memory each
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

struct BlockPoolGeom {
  int64_t block_bytes;        // P * R: one (page, layer) block
  int64_t row_bytes;          // R: device slot stride
  int64_t stage_page_stride;  // staging bytes from one page's block to the next page's
  int64_t max_d0;             // largest valid first device slot of a page (slots - P)
  int32_t page_size;
  uint32_t chunks;            // bulk copies per block
};

struct BlockSegment {
  char* dev;    // device layer buffer of this (pool, tensor, layer)
  char* stage;  // this (pool, tensor, layer)'s block of the launch's first page in staging
  int32_t pool;
  int32_t pad;
};

template <int MAXSEG>
struct BlockParams {
  static constexpr int kMaxSeg = MAXSEG;
  const void* dev_idx;  // device slot of every pair (device-visible)
  uint32_t* err;        // optional error word
  int64_t pair_begin;   // first pair of the launch's first page
  int32_t nseg;
  int32_t dir;          // kDevToPaged: device -> staging; kPagedToDev: staging -> device
  BlockPoolGeom pool[kMaxPools];
  int64_t seg_item_begin[MAXSEG + 1];  // items (chunks) before each segment
  BlockSegment seg[MAXSEG];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar` to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_test(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// At most one bulk-store group may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename IdxT>
__device__ __forceinline__ int64_t block_index(const void* base, int64_t i) {
  return static_cast<int64_t>(static_cast<const IdxT*>(base)[i]);
}

// Source, destination and size of chunk `item`; false (and an error bit) when
// its page's first device slot is out of range or an address is not 16-aligned.
template <typename IdxT, int MAXSEG>
__device__ __forceinline__ bool resolve(const BlockParams<MAXSEG>& p, int64_t item,
                                        const char** src, char** dst, uint32_t* bytes) {
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seg_item_begin[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const BlockSegment sg = p.seg[lo];
  const BlockPoolGeom& g = p.pool[sg.pool];
  const int64_t t = item - p.seg_item_begin[lo];
  const int64_t page = t / g.chunks;
  const int64_t off = (t - page * g.chunks) * int64_t(kChunk);
  *bytes = uint32_t(min(int64_t(kChunk), g.block_bytes - off));
  const int64_t d0 = block_index<IdxT>(p.dev_idx, p.pair_begin + page * g.page_size);
  if (d0 < 0 || d0 > g.max_d0) {
    if (p.err) atomicOr(p.err, HICACHE_DEVERR_RANGE);
    return false;
  }
  char* dev = sg.dev + d0 * g.row_bytes + off;
  char* stg = sg.stage + page * g.stage_page_stride + off;
  *src = p.dir == kDevToPaged ? dev : stg;
  *dst = p.dir == kDevToPaged ? stg : dev;
  if (((reinterpret_cast<uintptr_t>(*src) | reinterpret_cast<uintptr_t>(*dst) | *bytes) & 15u) != 0) {
    if (p.err) atomicOr(p.err, HICACHE_DEVERR_PAGE_ALIGN);
    return false;
  }
  return true;
}

// One resolved chunk: where it comes from, where it goes, how long it is
// (0 = skipped).
struct ChunkRef {
  const char* src;
  char* dst;
  uint32_t bytes;
};

template <typename IdxT, int MAXSEG>
__global__ void __launch_bounds__(32) page_block_kernel(const __grid_constant__ BlockParams<MAXSEG> p) {
  extern __shared__ __align__(128) unsigned char stage_buf[];
  __shared__ __align__(8) uint64_t bar[kStages];
  __shared__ char* dst_of[kStages];
  __shared__ uint32_t bytes_of[kStages];
  // Chunk tables of two batches of 32: the 32 lanes resolve a batch together
  // (one index load each, all in flight at once), lane 0 runs the copies.
  __shared__ ChunkRef table[2][32];
  const int lane = threadIdx.x;

  const int64_t nitems = p.seg_item_begin[p.nseg];
  const int64_t first = blockIdx.x;
  const int64_t step = gridDim.x;
  const int64_t K = first < nitems ? (nitems - first + step - 1) / step : 0;
  if (K == 0) return;

  auto resolve_batch = [&](int64_t b) {
    const int64_t k = b * 32 + lane;
    ChunkRef r{nullptr, nullptr, 0};
    if (k < K && !resolve<IdxT>(p, first + k * step, &r.src, &r.dst, &r.bytes)) r.bytes = 0;
    table[b & 1][lane] = r;
  };
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s]);
    mbar_init_fence();
  }
  resolve_batch(0);
  resolve_batch(1);
  __syncwarp();

  // Item k of this CTA goes through stage k % kStages.
  auto issue = [&](int64_t k) {
    const int s = int(k % kStages);
    const ChunkRef r = table[(k >> 5) & 1][k & 31];
    dst_of[s] = r.bytes ? r.dst : nullptr;
    bytes_of[s] = r.bytes;
    if (r.bytes) {
      mbar_expect_tx(&bar[s], r.bytes);
      bulk_load(stage_buf + size_t(s) * kChunk, r.src, r.bytes, &bar[s]);
    } else {
      mbar_arrive(&bar[s]);  // skipped: complete the stage's phase without data
    }
  };

  int64_t issued = 0;
  bool gave_up = false;
  if (lane == 0) {
    issued = K < kStages ? K : kStages;
    for (int64_t k = 0; k < issued; ++k) issue(k);
  }
  for (int64_t b = 0; b * 32 < K; ++b) {
    if (lane == 0 && !gave_up) {
      const int64_t kend = (b + 1) * 32 < K ? (b + 1) * 32 : K;
      for (int64_t k = b * 32; k < kend; ++k) {
        const int s = int(k % kStages);
        if (!mbar_wait(&bar[s], uint32_t((k / kStages) & 1))) {
          // Give up: report, let the loads still in flight land (bounded),
          // and let every store finish before the shared memory goes away.
          if (p.err) atomicOr(p.err, HICACHE_DEVERR_TIMEOUT);
          for (int64_t j = k; j < issued; ++j)  // this item's load too
            mbar_wait(&bar[j % kStages], uint32_t((j / kStages) & 1));
          gave_up = true;
          break;
        }
        fence_async_smem();
        if (dst_of[s]) bulk_store(dst_of[s], stage_buf + size_t(s) * kChunk, bytes_of[s]);
        bulk_commit();
        // Refill the stage of item k - 1, whose store was issued one item
        // ago; that item is at most kStages - 1 past this batch, so its
        // entry is in the next batch's table, which is resolved.
        if (k >= 1 && issued < K) {
          bulk_wait_read_all_but_one();
          issue(issued);
          ++issued;
        }
      }
    }
    gave_up = __shfl_sync(0xffffffffu, gave_up, 0);
    if (gave_up) break;
    __syncwarp();
    resolve_batch(b + 2);  // batch b's entries are no longer read
    __syncwarp();
  }
  if (lane == 0) bulk_wait_all();
}

template <typename IdxT, int MAXSEG>
hicache_status block_kernel_ready() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64)
    return fail(HICACHE_ECUDA, "page block copy: no current device");
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(page_block_kernel<IdxT, MAXSEG>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStages * kChunk);
    if (e != cudaSuccess)
      return fail(HICACHE_ECUDA, std::string("cudaFuncSetAttribute(page block kernel): ") +
                                     cudaGetErrorName(e));
    done[dev] = true;
  }
  return HICACHE_OK;
}

template <typename IdxT, int MAXSEG>
hicache_status launch_block_params(const BlockParams<MAXSEG>& prm, const LaunchCfg& cfg,
                                   cudaStream_t stream) {
  const int64_t items = prm.seg_item_begin[prm.nseg];
  if (items <= 0) return HICACHE_OK;
  hicache_status st = block_kernel_ready<IdxT, MAXSEG>();
  if (st != HICACHE_OK) return st;
  const int max_ctas = cfg.max_ctas > 0 ? cfg.max_ctas : device_sm_count() * kBlockCtasPerSm;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items, max_ctas)));
  page_block_kernel<IdxT, MAXSEG><<<grid, 32, kStages * kChunk, stream>>>(prm);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(HICACHE_ECUDA, std::string("page block kernel launch: ") + cudaGetErrorName(e));
  count_launch();
  return HICACHE_OK;
}

}  // namespace

bool page_blocks_ok(const PoolInfo& pi, const SideSpec& staging, size_t p) {
  const int64_t block = int64_t(pi.P) * pi.token_bytes;
  if (pi.layout != HICACHE_LAYOUT_PAGE_FIRST_DIRECT || block % 16 != 0) return false;
  // the first slot of a page lands on a 16-byte boundary: token rows of a
  // multiple of 16 bytes, or a page-granular pool whose pages start at
  // multiples of P
  if (pi.token_bytes % 16 != 0 && !pi.page_granular) return false;
  if (staging.layer_stride[p] != block || staging.page_stride[p] % 16 != 0) return false;
  for (char* d : pi.dev)
    if (reinterpret_cast<uintptr_t>(d) % 16 != 0) return false;
  for (char* b : staging.base[p])
    if (reinterpret_cast<uintptr_t>(b) % 16 != 0) return false;
  return true;
}

hicache_status load_block_kernels() {
  hicache_status st = block_kernel_ready<int32_t, kMaxSegSmall>();
  if (st == HICACHE_OK) st = block_kernel_ready<int32_t, kMaxSegLarge>();
  if (st == HICACHE_OK) st = block_kernel_ready<int64_t, kMaxSegSmall>();
  if (st == HICACHE_OK) st = block_kernel_ready<int64_t, kMaxSegLarge>();
  return st;
}

hicache_status launch_page_blocks(const std::vector<PoolInfo>& pools, const SideSpec& staging,
                                  const void* dev_idx, int32_t index_bits, int64_t page_begin,
                                  int64_t pages, Dir dir, int32_t layer_begin, int32_t layer_end,
                                  const LaunchCfg& cfg, cudaStream_t stream) {
  if (pages <= 0 || layer_end <= layer_begin) return HICACHE_OK;
  const int32_t P = pools[0].P;
  int32_t segs_per_layer = 0;
  for (const PoolInfo& pi : pools) segs_per_layer += pi.T;
  const bool small = int64_t(layer_end - layer_begin) * segs_per_layer <= kMaxSegSmall;

  auto run = [&](auto& prm) -> hicache_status {
    using Prm = std::remove_reference_t<decltype(prm)>;
    constexpr int kMax = Prm::kMaxSeg;
    prm.dev_idx = dev_idx;
    prm.err = cfg.err;
    prm.pair_begin = page_begin * P;
    prm.dir = dir;
    for (size_t p = 0; p < pools.size(); ++p) {
      const PoolInfo& pi = pools[p];
      BlockPoolGeom& g = prm.pool[p];
      g.block_bytes = int64_t(pi.P) * pi.token_bytes;
      g.row_bytes = pi.token_bytes;
      g.stage_page_stride = staging.page_stride[p];
      g.max_d0 = pi.device_slots - pi.P;
      g.page_size = pi.P;
      g.chunks = uint32_t((g.block_bytes + kChunk - 1) / kChunk);
    }
    int nseg = 0;
    int64_t items = 0;
    auto flush = [&]() -> hicache_status {
      prm.nseg = nseg;
      prm.seg_item_begin[nseg] = items;
      const hicache_status st = index_bits == 32
                                    ? launch_block_params<int32_t, kMax>(prm, cfg, stream)
                                    : launch_block_params<int64_t, kMax>(prm, cfg, stream);
      nseg = 0;
      items = 0;
      return st;
    };
    for (int32_t l = layer_begin; l < layer_end; ++l) {
      if (nseg + segs_per_layer > kMax) {
        const hicache_status st = flush();
        if (st != HICACHE_OK) return st;
      }
      for (size_t p = 0; p < pools.size(); ++p) {
        const PoolInfo& pi = pools[p];
        for (int32_t t = 0; t < pi.T; ++t) {
          BlockSegment& s = prm.seg[nseg];
          s.dev = pi.dev[size_t(t) * pi.L + l];
          s.stage = staging.base[p][size_t(t)] +
                    int64_t(l - staging.layer_origin) * staging.layer_stride[p];
          s.pool = int32_t(p);
          s.pad = 0;
          prm.seg_item_begin[nseg] = items;
          items += pages * int64_t(prm.pool[p].chunks);
          ++nseg;
        }
      }
    }
    return nseg > 0 ? flush() : HICACHE_OK;
  };
  if (small) {
    BlockParams<kMaxSegSmall> prm{};
    return run(prm);
  }
  static thread_local BlockParams<kMaxSegLarge> prm_large;
  prm_large = BlockParams<kMaxSegLarge>{};
  return run(prm_large);
}

}  // namespace hk
