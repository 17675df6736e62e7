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
// Work decomposition: a warp task is about 2 KiB of one segment (one pool,
// tensor and layer; 4 KiB for a launch of few CTAs against the host pool):
// up to 128 rows, or one 2 KiB (4 KiB) part of a longer row.  Lane
// r loads the pairs of rows r, r + 32, ..., checks them and writes each row's
// source and destination byte offsets into the warp's table in shared memory.
// The task's rows are then treated as one flat array of VEC-byte chunks: lane
// k of an iteration copies chunk c0 + k, reading its row's offsets from the
// table.  Rows that are adjacent on both sides therefore produce fully
// coalesced 512-byte warp accesses whatever the row size, which is how
// contiguous index runs are merged without any run table.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <mutex>
#include <numeric>
#include <string>

#include "consumer_kernel.cuh"
#include "hicache_internal.h"
#include "row_copy_kernel.cuh"

namespace hk {

namespace {

hicache_status cuda_fail(cudaError_t e, const char* what) {
  return fail(HICACHE_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                 cudaGetErrorString(e) + ")");
}

// CTAs a launch may use: the caller's cap, else the direction's default.
int cta_budget(const LaunchCfg& cfg, Dir dir) {
  if (cfg.max_ctas > 0) return cfg.max_ctas;
  const int sms = device_sm_count();
  if (cfg.paged_in_hbm) return sms * kCtasPerSmHbm;
  return dir == kDevToPaged ? sms * kCtasPerSmToHost : std::max(1, sms / kSmsPerCtaFromHost);
}

template <int MAXSEG, bool SIGNAL>
hicache_status launch_segments(const CopyParams<MAXSEG>& prm, int32_t index_bits, int64_t ntasks,
                               const LaunchCfg& cfg, bool deep, cudaStream_t stream) {
  if (ntasks <= 0) return HICACHE_OK;
  bool layer_rows = false, deep4 = false;
  for (int p = 0; p < kMaxPools; ++p) {
    layer_rows = layer_rows || prm.pool[p].layer_rows;
    deep4 = deep4 || prm.pool[p].vec == 4;
  }
  // 16-warp CTAs under a small cap (the layer-row instances keep 8 warps)
  const bool wide = deep && !layer_rows && cfg.max_ctas > 0 && cfg.max_ctas <= kWideMaxCtas;
  const int warps = wide ? kWarpsPerCtaWide : kWarpsPerCta;
  const int max_ctas = cta_budget(cfg, static_cast<Dir>(prm.dir));
  const int64_t want = (ntasks + warps - 1) / warps;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, max_ctas)));
  // one instance per index width, signalling, layer rows, 4-byte chunks, task
  // depth and CTA width
  auto go = [&](auto idx_tag, auto lr_tag, auto d4_tag) {
    using IdxT = decltype(idx_tag);
    constexpr bool LR = decltype(lr_tag)::value, D4 = decltype(d4_tag)::value;
    if constexpr (!LR) {
      if (wide) {
        row_copy_kernel<IdxT, MAXSEG, SIGNAL, false, D4, true, kWarpsPerCtaWide>
            <<<grid, kWarpsPerCtaWide * 32, 0, stream>>>(prm);
        return;
      }
    }
    if (deep)
      row_copy_kernel<IdxT, MAXSEG, SIGNAL, LR, D4, true, kWarpsPerCta>
          <<<grid, kThreadsPerCta, 0, stream>>>(prm);
    else
      row_copy_kernel<IdxT, MAXSEG, SIGNAL, LR, D4, false, kWarpsPerCta>
          <<<grid, kThreadsPerCta, 0, stream>>>(prm);
  };
  using F = std::false_type;
  using T = std::true_type;
  auto pick = [&](auto idx_tag) {
    if constexpr (SIGNAL) {
      if (deep4) go(idx_tag, F{}, T{}); else go(idx_tag, F{}, F{});
    } else if (layer_rows) {
      // the layer-row path runs 4-byte chunks deep by itself; the other pools
      // of such a launch take the shallow loop (a deep one measured slower)
      go(idx_tag, T{}, F{});
    } else {
      if (deep4) go(idx_tag, F{}, T{}); else go(idx_tag, F{}, F{});
    }
  };
  if (index_bits == 32) pick(int32_t{});
  else pick(int64_t{});
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "row copy kernel launch");
  count_launch();
  return HICACHE_OK;
}

}  // namespace

namespace {
std::atomic<int64_t> g_launches{0};

template <typename IdxT, int MAXSEG, bool LAYER_ROWS, bool DEEP4>
cudaError_t load_static_instance() {
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(
      &a, row_copy_kernel<IdxT, MAXSEG, false, LAYER_ROWS, DEEP4, false, kWarpsPerCta>);
  if (e == cudaSuccess)
    e = cudaFuncGetAttributes(
        &a, row_copy_kernel<IdxT, MAXSEG, false, LAYER_ROWS, DEEP4, true, kWarpsPerCta>);
  if constexpr (!LAYER_ROWS) {
    if (e == cudaSuccess)
      e = cudaFuncGetAttributes(
          &a, row_copy_kernel<IdxT, MAXSEG, false, false, DEEP4, true, kWarpsPerCtaWide>);
  }
  return e;
}

template <typename IdxT, int MAXSEG>
cudaError_t load_static_instances() {
  cudaError_t e = load_static_instance<IdxT, MAXSEG, false, false>();
  if (e == cudaSuccess) e = load_static_instance<IdxT, MAXSEG, false, true>();
  if (e == cudaSuccess) e = load_static_instance<IdxT, MAXSEG, true, false>();
  return e;
}
}  // namespace

hicache_status load_staged_backup_kernels() {
  // Under CUDA's lazy module loading a kernel is loaded, and its code placed
  // in device memory, at its first use; querying its attributes is such a use.
  cudaError_t e = load_static_instances<int32_t, kMaxSegSmall>();
  if (e == cudaSuccess) e = load_static_instances<int32_t, kMaxSegLarge>();
  if (e == cudaSuccess) e = load_static_instances<int64_t, kMaxSegSmall>();
  if (e == cudaSuccess) e = load_static_instances<int64_t, kMaxSegLarge>();
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(row copy kernel)");
  return load_block_kernels();
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

bool moves_page_rows(const PoolInfo& pi) {
  return pi.page_granular && pi.layout == HICACHE_LAYOUT_PAGE_FIRST_DIRECT;
}

int64_t moved_row_bytes(const PoolInfo& pi) {
  return moves_page_rows(pi) ? pi.token_bytes * pi.P : pi.token_bytes;
}

SideSpec host_side(const std::vector<PoolInfo>& pools) {
  SideSpec s;
  s.layer_origin = 0;
  for (const PoolInfo& pi : pools) {
    const bool direct = pi.layout == HICACHE_LAYOUT_PAGE_FIRST_DIRECT;
    // direct: [page][layer][token][row]; page_first: [token][layer][row]
    const int64_t layer_stride = direct ? int64_t(pi.P) * pi.token_bytes : pi.token_bytes;
    s.base.push_back(pi.host);
    s.layer_stride.push_back(layer_stride);
    s.page_stride.push_back(direct ? int64_t(pi.L) * pi.P * pi.token_bytes
                                   : int64_t(pi.L) * pi.token_bytes);
    s.rows_per_page.push_back(direct ? (moves_page_rows(pi) ? 1 : pi.P) : 1);
    s.paged_tokens.push_back(pi.host_pages * pi.P);
    s.vec16.push_back(vec16_ok(pi, pi.host, layer_stride));
  }
  return s;
}

bool vec16_ok(const PoolInfo& pi, const std::vector<char*>& paged_bases, int64_t layer_stride) {
  if (moved_row_bytes(pi) % 16 != 0 || layer_stride % 16 != 0) return false;
  for (char* ptr : pi.dev)
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
  for (char* ptr : paged_bases)
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
  return true;
}

void fill_geometry(const PoolInfo& pi, int64_t npairs, int vec, int64_t paged_page_stride,
                   int64_t paged_tokens, int32_t rows_per_page, int64_t task_bytes, int unroll16,
                   bool fill_rows, PoolGeom* g) {
  const int64_t R = moved_row_bytes(pi);
  const bool page_rows = moves_page_rows(pi);
  g->row_bytes = R;
  g->paged_page_stride = paged_page_stride;
  g->dev_tokens = pi.device_slots;
  g->paged_tokens = paged_tokens;
  g->rows_per_page = rows_per_page;
  g->idx_stride = page_rows ? pi.P : 1;
  g->idx_div = page_rows ? pi.P : 1;
  g->nrows = page_rows ? npairs / pi.P : npairs;
  g->vec = uint32_t(vec);
  g->cpr = uint32_t(R / vec);
  g->q32 = 32u / g->cpr;
  g->r32 = 32u % g->cpr;
  g->qS = uint32_t(32 * kUnroll) / g->cpr;
  g->rS = uint32_t(32 * kUnroll) % g->cpr;
  // about task_bytes per task (2 KiB, or 4 KiB for deep tasks): 128 rows of
  // 16 B, one row of 2 KiB, or one 2 KiB part of a longer row (a state slot of
  // several MiB, a long page row).
  // The row count is rounded up so that a task spans whole 128-byte lines when
  // its rows are contiguous (a run of whole pages starts on a line): a line
  // that two warps write at different times reaches the host in two partial
  // writes.  Rows whose bytes already fill lines (2 KiB, 1152 B) keep their count.
  int64_t rpt = (task_bytes + R - 1) / R;
  if (R <= task_bytes) {
    const int64_t line_rows = 128 / std::gcd(R, int64_t(128));  // rows that fill whole lines
    const int64_t rounded = (rpt + line_rows - 1) / line_rows * line_rows;
    if (rounded <= kMaxRowsPerTask) rpt = rounded;
    if (vec == 16 && fill_rows) {
      // The copy loop moves 32 * unroll16 chunks per iteration, one host-link
      // round trip each.  Among the row counts that keep whole lines and at
      // most two iterations, a count that fills the iterations' chunks better
      // replaces the target: 1152-byte rows (72 chunks) fill 56 % of two deep
      // iterations at 4 rows and 98 % at 7, 56 % of two shallow ones at 2 rows
      // and 84 % at 3.
      const int64_t cpr = R / 16;
      const int64_t slots = 32 * int64_t(unroll16);
      auto fill = [&](int64_t k) {
        const int64_t c = k * cpr;
        return double(c) / double((c + slots - 1) / slots * slots);
      };
      double best = fill(rpt);
      for (int64_t k = line_rows; k <= kMaxRowsPerTask && k * cpr <= 2 * slots; k += line_rows) {
        if (fill(k) > best + 1e-9) {
          best = fill(k);
          rpt = k;
        }
      }
    }
  }
  g->rows_per_task = int32_t(std::min<int64_t>(kMaxRowsPerTask, std::max<int64_t>(1, rpt)));
  g->part_chunks = uint32_t(task_bytes / vec);
  g->parts_per_row = R > task_bytes ? int32_t((g->cpr + g->part_chunks - 1) / g->part_chunks) : 1;
  g->tasks_per_seg = g->parts_per_row > 1
                         ? g->nrows * g->parts_per_row
                         : (g->nrows + g->rows_per_task - 1) / g->rows_per_task;
  g->layer_rows = 0;
  g->num_layers = 0;
  g->seg_stride = 0;
  g->tasks_per_token = 0;
  g->tokens_per_task = 0;
}

hicache_status launch_rows(const std::vector<PoolInfo>& pools, const SideSpec& side,
                           const void* dev_idx, const void* paged_idx, int32_t index_bits,
                           int64_t pair_begin, int64_t npairs, Dir dir, int32_t layer_begin,
                           int32_t layer_end, const LaunchCfg& cfg, cudaStream_t stream,
                           const BurstWords* signal) {
  if (npairs <= 0 || layer_end <= layer_begin) return HICACHE_OK;
  int32_t segs_per_layer = 0;
  for (const PoolInfo& pi : pools) segs_per_layer += pi.T;
  const bool small =
      !signal && int64_t(layer_end - layer_begin) * segs_per_layer <= kMaxSegSmall;

  // Deep tasks for a launch against the host pool with few CTAs.
  const bool deep = !cfg.paged_in_hbm && cta_budget(cfg, dir) <= kDeepMaxCtas;
  const int64_t task_bytes = deep ? kTaskBytesDeep : kTaskBytes;
  // Rows per task chosen to fill the copy loop's iterations, except for a
  // load at its default budget: there the link is full either way, and the
  // larger tasks measured a longer lag for a consumer gated by the layer
  // events (78-layer: 92 against 57 us after its event).
  const bool fill_rows = !(deep && cfg.max_ctas <= 0);
  auto run = [&](auto& prm, int maxseg) -> hicache_status {
    prm.dev_idx = dev_idx;
    prm.paged_idx = paged_idx;
    prm.err = cfg.err;
    prm.dir = dir;
    prm.pair_begin = pair_begin;
    int64_t tasks_per_layer = 0;
    const bool one_launch = int64_t(layer_end - layer_begin) * segs_per_layer <= maxseg;
    for (size_t p = 0; p < pools.size(); ++p) {
      const PoolInfo& pi = pools[p];
      PoolGeom& g = prm.pool[p];
      fill_geometry(pi, npairs, side.vec16[p] ? 16 : 4, side.page_stride[p],
                    side.paged_tokens[p], side.rows_per_page[p], task_bytes,
                    deep ? kUnrollDeep : kUnroll, fill_rows, &g);
      // An all-layer backup into a token-major host pool whose rows do not fill
      // whole lines: one task per token and up to kMaxRowsPerTask of its
      // layers, which are adjacent on the host, instead of rows of one layer
      // that each cover lines in part.
      const int64_t R = pi.token_bytes;
      if (dir == kDevToPaged && !signal && !cfg.paged_in_hbm && one_launch &&
          layer_begin == 0 && layer_end == pi.L && !moves_page_rows(pi) &&
          side.rows_per_page[p] == 1 && side.layer_stride[p] == R &&
          side.page_stride[p] == int64_t(pi.L) * R && R <= task_bytes && R % 128 != 0) {
        g.layer_rows = 1;
        g.num_layers = pi.L;
        g.seg_stride = segs_per_layer;
        // about task_bytes of adjacent host rows per task: several tokens when
        // a token's layers hold less, part of a token when it has more than
        // kMaxRowsPerTask layers
        const int64_t per_token = int64_t(pi.L) * R;
        const int64_t kt = std::min<int64_t>(std::max<int64_t>(1, (task_bytes + per_token - 1) / per_token),
                                             std::max<int64_t>(1, kMaxRowsPerTask / pi.L));
        g.tokens_per_task = int32_t(kt);
        g.rows_per_task = pi.L >= kMaxRowsPerTask ? kMaxRowsPerTask : int32_t(kt) * pi.L;
        g.tasks_per_token = (pi.L + g.rows_per_task - 1) / g.rows_per_task;  // 1 unless L > 128
        g.tasks_per_seg = g.tasks_per_token > 1 ? g.nrows * g.tasks_per_token
                                                : (g.nrows + kt - 1) / kt;  // all on layer 0's segment
      }
      tasks_per_layer += int64_t(pi.T) * g.tasks_per_seg;
    }
    // A signalling launch covers whole groups of layers only and counts a
    // group's tasks in a 32-bit word; one group must fit in one launch.
    const int32_t lpg = signal ? std::max<int32_t>(1, signal->layers_per_group) : 1;
    if (signal && tasks_per_layer * lpg > kMaxSignalTasks)
      return fail(HICACHE_EINVAL, "single-launch burst: more than 2^30 tasks in one layer group");
    const int cap = signal ? (maxseg / segs_per_layer) * segs_per_layer : maxseg;
    if (signal && int64_t(lpg) * segs_per_layer > cap)
      return fail(HICACHE_EINVAL, "single-launch burst: a layer group is larger than one launch");
    int nseg = 0;
    int64_t tasks = 0;
    int32_t first_layer = layer_begin;
    auto flush = [&](int32_t next_layer) -> hicache_status {
      prm.nseg = nseg;
      prm.seg_task_begin[nseg] = tasks;
      hicache_status st;
      if (signal) {
        prm.sig.done = signal->done;
        prm.sig.flag = signal->flag;
        prm.sig.exits = signal->exits;
        prm.sig.next = signal->next;
        prm.sig.tasks_per_layer = tasks_per_layer;
        prm.sig.segs_per_layer = segs_per_layer;
        prm.sig.layer_base = first_layer - layer_begin;
        prm.sig.nlayers = next_layer - first_layer;
        prm.sig.layers_per_group = lpg;
        prm.sig.burst_layers = layer_end - layer_begin;
        st = launch_segments<std::remove_reference_t<decltype(prm)>::kMaxSeg, true>(
            prm, index_bits, tasks, cfg, deep, stream);
      } else {
        st = launch_segments<std::remove_reference_t<decltype(prm)>::kMaxSeg, false>(
            prm, index_bits, tasks, cfg, deep, stream);
      }
      nseg = 0;
      tasks = 0;
      first_layer = next_layer;
      return st;
    };
    for (int32_t l = layer_begin; l < layer_end; ++l) {
      // a launch is cut only where a group starts, when the whole group
      // would not fit
      if ((l - layer_begin) % lpg == 0) {
        const int64_t gl = std::min<int32_t>(lpg, layer_end - l);
        if (nseg + gl * segs_per_layer > cap ||
            (signal && nseg > 0 && tasks + gl * tasks_per_layer > kMaxSignalTasks)) {
          const hicache_status st = flush(l);
          if (st != HICACHE_OK) return st;
        }
      }
      for (size_t p = 0; p < pools.size(); ++p) {
        const PoolInfo& pi = pools[p];
        for (int32_t t = 0; t < pi.T; ++t) {
          Segment& s = prm.seg[nseg];
          s.dev = pi.dev[size_t(t) * pi.L + l];
          s.paged = side.base[p][size_t(t)] + int64_t(l - side.layer_origin) * side.layer_stride[p];
          s.pool = int32_t(p);
          s.pad = 0;
          prm.seg_task_begin[nseg] = tasks;
          // a layer-row pool's tasks all belong to its layer-0 segment
          if (!prm.pool[p].layer_rows || l == layer_begin) tasks += prm.pool[p].tasks_per_seg;
          ++nseg;
        }
      }
    }
    return nseg > 0 ? flush(layer_end) : HICACHE_OK;
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
  const int grid = int(std::min<int64_t>((n + kWarpsPerCta - 1) / kWarpsPerCta,
                                         int64_t(device_sm_count()) * 4));
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
