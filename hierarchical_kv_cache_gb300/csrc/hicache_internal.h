// hicache_internal.h -- types shared by the library's translation units.
//
// Nothing here is part of the public ABI (include/hicache.h is).  The copy
// kernels see a transfer as a list of "segments": one segment is the stream of
// rows of one (pool, tensor, layer) between a layer-first device buffer and the
// page-first host tensor (or an HBM staging buffer laid out like it).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include <cuda_runtime_api.h>

#include "hicache.h"

namespace hk {

constexpr int kMaxPools = 4;
constexpr int kWarpsPerCta = 8;     // 256-thread CTAs
constexpr int kThreadsPerCta = kWarpsPerCta * 32;
constexpr int kUnroll = 4;          // chunks in flight per lane per iteration
constexpr int kMaxRowsPerTask = 128; // rows of one warp task (shared-memory offset table)
constexpr int64_t kTaskBytes = 2048; // target payload of one warp task
// Deep tasks, for launches with few CTAs against the host pool: twice the
// payload per task and twice the chunks in flight per lane, so that each warp
// keeps twice the bytes outstanding on the host link.  Measured on GB300 with
// 16 CTAs: a Llama-3-8B burst 157 against 93 GB/s, a 78-layer backup 177
// against 117.  With one CTA per SM they cost a concurrent GEMM more (their
// registers crowd it out: 39 against 27 % during a burst) and move no more, so
// launches of more than kDeepMaxCtas CTAs keep the shallow tasks.
constexpr int kUnrollDeep = 8;
constexpr int64_t kTaskBytesDeep = 4096;
constexpr int kDeepMaxCtas = 76;
// Wide CTAs, for launches the caller caps at kWideMaxCtas CTAs or fewer: 16
// warps of deep tasks per CTA instead of 8, so that the few SMs such a cap
// allows keep twice the bytes in flight.  Measured on GB300 beside a bf16 GEMM
// loop, 8 CTAs: a 78-layer backup 158 against 77 GB/s, its burst 139 against
// 69, the GEMM within 1.3 % or faster meanwhile; 16 CTAs: 178 against 157 and
// 196 against 142, the GEMM 2-5 % slower meanwhile over a shorter transfer.
// From 20 CTAs up 16 warps cost the GEMM more per byte moved than 8.  Up to
// 128 registers a thread fit 512 threads; the layer-row instances need more
// and keep 8 warps.
constexpr int kWarpsPerCtaWide = 16;
constexpr int kWideMaxCtas = 16;
constexpr int kMaxSegSmall = 8;     // per-layer launches: pools x tensors
constexpr int kMaxSegLarge = 512;   // all-layer launches: pools x tensors x layers
// A signalling launch hands out its tasks from a 32-bit counter that every warp
// bumps once past the last task; launches are cut at layer boundaries so that
// tasks plus claims stay far below 2^32 (2^30 tasks is about 2 TB of rows).
constexpr int64_t kMaxSignalTasks = int64_t(1) << 30;

// Direction of one launch.
enum Dir : int32_t { kDevToPaged = 0, kPagedToDev = 1 };

// Row geometry of one pool for one launch.  A "row" is what one pair moves:
// a token row (R bytes) for token pools, a whole page row (P * R bytes) for
// page-granular pools.
struct PoolGeom {
  int64_t row_bytes;         // bytes moved per row
  int64_t paged_page_stride; // bytes from one page of the paged side to the next
  int64_t dev_tokens;        // token rows of one device layer buffer (range check)
  int64_t paged_tokens;      // token rows of the paged side (range check)
  int64_t nrows;             // rows moved by one segment of this pool
  int64_t tasks_per_seg;     // ceil(nrows / rows_per_task), or nrows * parts_per_row
  int32_t rows_per_page;     // P for token pools, 1 for page-granular pools
  int32_t idx_stride;        // pair index of row k is k * idx_stride (P for page pools)
  int32_t idx_div;           // token index -> row index divisor (P for page pools)
  int32_t rows_per_task;     // 1..kMaxRowsPerTask rows handled by one warp task
  uint32_t cpr;              // chunks (vec bytes) per row
  uint32_t q32, r32;         // 32 == q32 * cpr + r32
  uint32_t qS, rS;           // 32 * kUnroll == qS * cpr + rS
  uint32_t vec;              // chunk bytes: 16, or 4 when a row or base is not 16-aligned
  int32_t parts_per_row;     // > 1: a row longer than a task is split into this many tasks
  uint32_t part_chunks;      // chunks of one such part (the last part may be shorter)
  // Layer rows (all-layer backup into a token-major host pool): a task moves
  // layers [k * rows_per_task, ...) of one token, whose layers are adjacent on
  // the host, so that its host writes cover whole lines.  Its rows are layers;
  // every task of the (pool, tensor) belongs to its layer-0 segment, and layer
  // l's device buffer is the one of segment (that segment + l * seg_stride).
  // A token whose layers hold little (L * R well under a task) shares a task
  // with the next tokens: row f of such a task is layer f % L of its token f / L.
  int32_t layer_rows;        // 1 = this mode
  int32_t num_layers;        // L (layer rows only)
  int32_t seg_stride;        // segments from one layer to the next (layer rows only)
  int32_t tasks_per_token;   // ceil(L / rows_per_task) when a token spans tasks, else 1
  int32_t tokens_per_task;   // tokens sharing a task (1 when a token spans tasks)
};

// One (pool, tensor, layer) stream.
struct Segment {
  char* dev;    // device layer buffer base
  char* paged;  // paged-side base of this layer: host tensor (or staging) + layer block offset
  int32_t pool;
  int32_t pad;
};

// Completion signalling of a single-launch burst, per group of consecutive
// layers.  Segments are ordered layer-major, segs_per_layer per layer; layer k
// of the launch is burst layer layer_base + k, in group (layer_base + k) /
// layers_per_group.  A launch starts on a group boundary.  Words (device
// memory, zeroed before the launch): done[group] counts finished tasks,
// flag[group] becomes 1 once every task of that group's layers has landed;
// exits[launch first layer] counts CTAs that left the launch and
// next[launch first layer] hands out its tasks.  Groups are one layer for
// layers of 2 MiB or more, so a consumer can start on each as it lands, and
// several small layers otherwise, so the burst pays its stream waits per
// group rather than per layer.
struct SignalSpec {
  uint32_t* done = nullptr;
  uint32_t* flag = nullptr;
  uint32_t* exits = nullptr;
  uint32_t* next = nullptr;
  int64_t tasks_per_layer = 0;
  int32_t segs_per_layer = 0;
  int32_t layer_base = 0;        // burst-relative index of this launch's first layer
  int32_t nlayers = 0;           // layers covered by this launch
  int32_t layers_per_group = 1;  // layers counted by one done/flag word
  int32_t burst_layers = 0;      // signalled layers of the whole burst (all launches)
  int32_t pad = 0;
};

template <int MAXSEG>
struct CopyParams {
  static constexpr int kMaxSeg = MAXSEG;
  const void* dev_idx;      // device-slot indices (device-accessible)
  const void* paged_idx;    // paged-side token indices; NULL = pair index - pair_begin
  uint32_t* err;            // optional device-accessible error word
  int64_t pair_begin;       // first pair moved by this launch
  int32_t nseg;
  int32_t dir;              // Dir
  SignalSpec sig;           // unused unless the kernel is the signalling instance
  PoolGeom pool[kMaxPools];
  int64_t seg_task_begin[MAXSEG + 1];
  Segment seg[MAXSEG];
};

// Host-side description of one validated pool.
struct PoolInfo {
  int32_t L, T, P;
  int32_t page_granular;
  int32_t layout;           // hicache_layout of the host tensors
  int64_t token_bytes;      // R of one token row
  int64_t device_slots, host_pages;
  std::vector<char*> dev;   // T * L device layer pointers
  std::vector<char*> host;  // T host tensor pointers (device-visible addresses)
};

// The two index arrays of a call: addresses the kernels use and, for host-located
// indices, addresses the CPU reads (NULL for device-located indices).
struct IndexSet {
  const void* dev_gpu = nullptr;
  const void* host_gpu = nullptr;
  const void* dev_cpu = nullptr;
  const void* host_cpu = nullptr;
  int32_t bits = 64;
  int64_t n = 0;
};

// Per-thread last error message.
void set_error(const std::string& msg);
void clear_error();
hicache_status fail(hicache_status st, const std::string& msg);

// Validation helpers (validate.cpp).
hicache_status check_pools(const hicache_pool* pools, int32_t num_pools, std::vector<PoolInfo>* out);
hicache_status check_index_args(const void* a, const void* b, int32_t index_bits, int64_t n);
// Range, distinct destinations and page-granular whole pages, on host-readable indices.
// dest_is_device selects which side must be distinct.
hicache_status check_pairs_host(const std::vector<PoolInfo>& pools, const void* dev_idx,
                                const void* host_idx, int32_t index_bits, int64_t n,
                                bool dest_is_device);
hicache_status plan_runs(const void* dev_idx, const void* host_idx, int32_t index_bits, int64_t n,
                         int32_t page_size, hicache_run* runs, int64_t cap, int64_t* num_runs,
                         int64_t* full_pages);

// Launch-side helpers (zero_copy.cu).
// Default CTAs of a copy launch (256 threads each).  Measured on GB300:
// one CTA per SM reaches the host-link peak in either direction alone (two
// per SM moved no more: 210.3 against 210.4 GB/s for a 32-layer burst).
// Beside compute the count matters: with a bf16 GEMM loop running, a burst of
// two CTAs per SM cost the GEMM 59-64 % of its throughput during the burst,
// one per SM 26-34 %, at the same transfer speed.  A load (host to device)
// defaults to one CTA per two SMs, which takes the deep tasks: it still moved
// 210-211 GB/s on every benchmark workload, and cost the GEMM 17-27 %.  A
// backup keeps one CTA per SM: with the deep tasks at one per two SMs a
// Llama-3-8B backup moved 190.7 against 193.3 GB/s (a 78-layer one 189.1
// against 192.4 in another run).  A caller that runs a backup and a load-back
// at once gets the most from the shared link with 76 deep CTAs on both sides
// (opts.max_ctas = 76: 298-317 GB/s together, against 245 with the defaults
// and 240 with two CTAs per SM each).  The staged path's
// gather and scatter row kernels (between the device pool and HBM staging,
// overlapped with copy-engine DMA) take two per SM.
constexpr int kCtasPerSmToHost = 1;
constexpr int kSmsPerCtaFromHost = 2;
constexpr int kCtasPerSmHbm = 2;

struct LaunchCfg {
  int max_ctas;   // 0 = default for the direction
  uint32_t* err;
  bool paged_in_hbm = false;  // the paged side is an HBM staging buffer
};

// The page-first side of a launch: the pinned host pool, or an HBM staging
// buffer laid out the same way.  Indexed [pool] and [pool][tensor].
struct SideSpec {
  std::vector<bool> vec16;                // [pool] 16-byte chunks usable on both sides
  int32_t layer_origin = 0;               // layer whose block starts at base
  std::vector<std::vector<char*>> base;   // [pool][tensor] base address
  std::vector<int64_t> layer_stride;      // [pool] bytes between layer blocks of one page
  std::vector<int64_t> page_stride;       // [pool] bytes between pages
  std::vector<int64_t> paged_tokens;      // [pool] token rows addressable on this side
  std::vector<int32_t> rows_per_page;     // [pool] rows between page strides on this side
};

// True when the pool moves whole page rows (page-granular pool, direct layout).
bool moves_page_rows(const PoolInfo& pi);
int64_t moved_row_bytes(const PoolInfo& pi);
// The host pool as a paged side, for either host layout.
SideSpec host_side(const std::vector<PoolInfo>& pools);
// 16-byte chunks are usable for pool `pi` against paged-side bases `paged_bases`
// whose layer blocks are `layer_stride` bytes apart.
bool vec16_ok(const PoolInfo& pi, const std::vector<char*>& paged_bases, int64_t layer_stride);
// task_bytes and unroll16: kTaskBytes and kUnroll, or kTaskBytesDeep and
// kUnrollDeep for a launch of deep tasks.  fill_rows: choose the rows per task
// that fill the copy loop's iterations (else the count nearest task_bytes).
void fill_geometry(const PoolInfo& pi, int64_t npairs, int vec, int64_t paged_page_stride,
                   int64_t paged_tokens, int32_t rows_per_page, int64_t task_bytes, int unroll16,
                   bool fill_rows, PoolGeom* g);
// Moves pairs [pair_begin, pair_begin + npairs) for layers [layer_begin, layer_end)
// of every pool and tensor between the device buffers and `side`.  With
// `signal` (words of a single-launch burst: done and flag indexed by group
// (l - layer_begin) / layers_per_group, exits and next by l - layer_begin),
// launches are cut at group boundaries and every group's flag word is set once
// all of its rows have landed.
struct BurstWords {
  uint32_t* done = nullptr;
  uint32_t* flag = nullptr;
  uint32_t* exits = nullptr;
  uint32_t* next = nullptr;
  int32_t layers_per_group = 1;  // launches are cut only at multiples of this many layers
};
hicache_status launch_rows(const std::vector<PoolInfo>& pools, const SideSpec& side,
                           const void* dev_idx, const void* paged_idx, int32_t index_bits,
                           int64_t pair_begin, int64_t npairs, Dir dir, int32_t layer_begin,
                           int32_t layer_end, const LaunchCfg& cfg, cudaStream_t stream,
                           const BurstWords* signal = nullptr);
// Page-block copies (block_copy.cu): whole (page, layer) blocks of P * R bytes
// between the device pool and HBM staging, with bulk-copy (TMA) loads and
// stores.  Usable for pool `p` of `staging` when page_blocks_ok holds and every
// page's P device slots are consecutive (checked by the caller).  Moves pages
// [page_begin, page_begin + pages) of the pair list (the pair of page k's
// first token is k * P) for layers [layer_begin, layer_end).
bool page_blocks_ok(const PoolInfo& pi, const SideSpec& staging, size_t p);
hicache_status launch_page_blocks(const std::vector<PoolInfo>& pools, const SideSpec& staging,
                                  const void* dev_idx, int32_t index_bits, int64_t page_begin,
                                  int64_t pages, Dir dir, int32_t layer_begin, int32_t layer_end,
                                  const LaunchCfg& cfg, cudaStream_t stream);
// Loads every instance of the page-block kernel on the current device.
hicache_status load_block_kernels();
hicache_status launch_checksum(const PoolInfo& pool, int32_t tensor, int32_t layer,
                               const void* dev_idx, int32_t index_bits, int64_t n,
                               uint64_t* out, cudaStream_t stream);
int device_sm_count();
// Loads, on the current device, every kernel instance that the staged
// all-layer backup can launch: the row-copy kernel with static striding (both
// index widths and segment capacities; 16- and 4-byte chunks; layer rows, for
// a small pool backed up zero-copy beside the staged ones) and the page-block
// kernel, so that later launches place no more code in device memory.
hicache_status load_staged_backup_kernels();
void count_launch();
int64_t kernel_launches();

}  // namespace hk
