// api.cu -- the extern "C" entry points declared in include/hicache.h.
//
// Each entry point validates everything on the host first (no copy is
// enqueued for a rejected call), resolves the device-visible addresses of the
// pinned host buffers, picks a path and enqueues the copies on the caller's
// stream.  Load calls record their layer-done events on every return path, the
// error convention of "[HiCache] Run the host->device load-back enqueue on a
// loader thread" (Modifications: a failed load completes every layer event).
#include <cuda_runtime.h>

#include <mutex>
#include <string>
#include <vector>

#include "burst.h"
#include "hicache_internal.h"
#include "staged.h"

namespace hk {
const std::string& last_error();

namespace {

hicache_opts default_opts() {
  hicache_opts o{};
  o.path = HICACHE_PATH_AUTO;
  o.index_location = HICACHE_INDEX_HOST;
  return o;
}

hicache_status check_opts(const hicache_opts& o) {
  if (o.path < HICACHE_PATH_AUTO || o.path > HICACHE_PATH_STAGED)
    return fail(HICACHE_EINVAL, "opts.path is not a hicache_path");
  if (o.index_location != HICACHE_INDEX_HOST && o.index_location != HICACHE_INDEX_DEVICE)
    return fail(HICACHE_EINVAL, "opts.index_location is not a hicache_index_location");
  if (o.max_ctas < 0) return fail(HICACHE_EINVAL, "opts.max_ctas is negative");
  if (o.reserved != 0) return fail(HICACHE_EINVAL, "opts.reserved must be 0");
  return HICACHE_OK;
}

hicache_status cuda_fail(cudaError_t e, const std::string& what) {
  return fail(HICACHE_ECUDA, what + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

enum class Want { kHostPinned, kDevice, kAny };

// Device-visible address of `ptr`, checking where it lives.
hicache_status device_view(const void* ptr, Want want, const std::string& what, const void** out) {
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "cudaPointerGetAttributes(" + what + ")");
  }
  const bool host = a.type == cudaMemoryTypeHost;
  const bool dev = a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
  if (want == Want::kHostPinned && !host)
    return fail(HICACHE_EINVAL, what + " must be pinned (page-locked) host memory");
  if (want == Want::kDevice && !dev) return fail(HICACHE_EINVAL, what + " must be device memory");
  if (!host && !dev)
    return fail(HICACHE_EINVAL, what + " is not memory the GPU can address (pin it first)");
  *out = (host && a.devicePointer) ? a.devicePointer : ptr;
  return HICACHE_OK;
}

// An optional buffer that kernels or stream operations write: NULL, or memory
// of kind `want` whose address is a multiple of `align`.  On success *ptr
// becomes its device-visible address.
template <typename T>
hicache_status check_gpu_buffer(T** ptr, Want want, size_t align, const std::string& what) {
  if (!*ptr) return HICACHE_OK;
  if (reinterpret_cast<uintptr_t>(*ptr) % align != 0)
    return fail(HICACHE_EALIGN, what + " is not " + std::to_string(align) + "-byte aligned");
  const void* v = nullptr;
  const hicache_status st = device_view(*ptr, want, what, &v);
  if (st != HICACHE_OK) return st;
  *ptr = static_cast<T*>(const_cast<void*>(v));
  return HICACHE_OK;
}

// True when `ptr` is device memory the CPU must not read.  When the query
// itself fails (no usable device, or memory CUDA does not know) it cannot be
// device memory of this process.
bool is_device_memory(const void* ptr) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

struct Prepared {
  std::vector<PoolInfo> pools;
  hicache_opts o{};
  IndexSet idx;
};

// Checks arguments and indices; resolves device-visible addresses.
size_t index_array_bytes(int64_t n, int32_t bits) {
  return (size_t(n) * size_t(bits / 8) + 15) / 16 * 16;
}

// With host-located indices and opts.index_staging, copies both validated index
// arrays into the staging buffer on `stream` and points the kernels at the copies.
hicache_status stage_indices(Prepared* pr, cudaStream_t stream) {
  const hicache_opts& o = pr->o;
  if (o.index_location != HICACHE_INDEX_HOST || !o.index_staging || pr->idx.n == 0)
    return HICACHE_OK;
  const size_t one = index_array_bytes(pr->idx.n, pr->idx.bits);
  if (o.index_staging_bytes < 2 * one)
    return fail(HICACHE_EINVAL, "opts.index_staging holds " + std::to_string(o.index_staging_bytes) +
                                    " bytes; this call needs " + std::to_string(2 * one));
  if (reinterpret_cast<uintptr_t>(o.index_staging) % 16 != 0)
    return fail(HICACHE_EALIGN, "opts.index_staging is not 16-byte aligned");
  char* dst = static_cast<char*>(o.index_staging);
  const size_t bytes = size_t(pr->idx.n) * size_t(pr->idx.bits / 8);
  cudaError_t e = cudaMemcpyAsync(dst, pr->idx.dev_cpu, bytes, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dst + one, pr->idx.host_cpu, bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(indices -> opts.index_staging)");
  pr->idx.dev_gpu = dst;
  pr->idx.host_gpu = dst + one;
  return HICACHE_OK;
}

// When check_layers is set, [layer_begin, layer_end) must lie inside the pools' layers.
hicache_status prepare(const hicache_pool* pools, int32_t num_pools, const void* dev_idx,
                       const void* host_idx, int32_t bits, int64_t n, const hicache_opts* opts,
                       bool dest_is_device, bool check_layers, int32_t layer_begin,
                       int32_t layer_end, Prepared* out) {
  out->o = opts ? *opts : default_opts();
  hicache_status st = check_pools(pools, num_pools, &out->pools);
  if (st != HICACHE_OK) return st;
  if (check_layers) {
    if (layer_begin < 0 || layer_end > out->pools[0].L || layer_begin > layer_end)
      return fail(HICACHE_EINVAL, "layer range [" + std::to_string(layer_begin) + ", " +
                                      std::to_string(layer_end) + ") outside the pools' " +
                                      std::to_string(out->pools[0].L) + " layers");
  }
  st = check_opts(out->o);
  if (st != HICACHE_OK) return st;
  st = check_index_args(dev_idx, host_idx, bits, n);
  if (st != HICACHE_OK) return st;
  out->idx.bits = bits;
  out->idx.n = n;
  if (out->o.index_location == HICACHE_INDEX_HOST) {
    // The CPU reads host-located indices next: they must not be device memory.
    if (n > 0 && (is_device_memory(dev_idx) || is_device_memory(host_idx)))
      return fail(HICACHE_EINVAL, "index_location is HICACHE_INDEX_HOST but an index array is "
                                  "device memory");
    out->idx.dev_cpu = dev_idx;
    out->idx.host_cpu = host_idx;
    st = check_pairs_host(out->pools, dev_idx, host_idx, bits, n, dest_is_device);
    if (st != HICACHE_OK) return st;
  }
  if (n == 0) return HICACHE_OK;
  // Host pool tensors: pinned memory (or device memory) the kernels can address.
  for (size_t p = 0; p < out->pools.size(); ++p) {
    for (size_t t = 0; t < out->pools[p].host.size(); ++t) {
      const void* v = nullptr;
      st = device_view(out->pools[p].host[t], Want::kAny,
                       "host tensor " + std::to_string(t) + " of pool " + std::to_string(p), &v);
      if (st != HICACHE_OK) return st;
      out->pools[p].host[t] = static_cast<char*>(const_cast<void*>(v));
    }
  }
  const Want w = out->o.index_location == HICACHE_INDEX_HOST ? Want::kHostPinned : Want::kDevice;
  st = device_view(dev_idx, w, "device_indices", &out->idx.dev_gpu);
  if (st != HICACHE_OK) return st;
  st = device_view(host_idx, w, "host_indices", &out->idx.host_gpu);
  if (st != HICACHE_OK) return st;
  if (out->o.path == HICACHE_PATH_STAGED &&
      (!out->o.staging[0] || !out->o.staging[1] || out->o.staging_bytes == 0))
    return fail(HICACHE_ENOSTAGE, "staged path requested without two staging buffers");
  // The optional buffers the copy writes: a pointer of the wrong kind or
  // alignment is an error status here, not a fault on the GPU later.
  hicache_opts& o = out->o;
  st = check_gpu_buffer(&o.device_error, Want::kAny, 4, "opts.device_error");
  if (st == HICACHE_OK) st = check_gpu_buffer(&o.burst_words, Want::kDevice, 4, "opts.burst_words");
  if (st == HICACHE_OK)
    st = check_gpu_buffer(&o.index_staging, Want::kDevice, 16, "opts.index_staging");
  for (int b = 0; b < 2 && st == HICACHE_OK; ++b)
    st = check_gpu_buffer(&o.staging[b], Want::kDevice, 16,
                          "opts.staging[" + std::to_string(b) + "]");
  return st;
}

// Host-only checks of opts->burst_words for a burst of `count` layers.
hicache_status check_burst_words(const hicache_opts& o, int32_t count) {
  if (!o.burst_words) return HICACHE_OK;
  if (o.burst_words_len < kBurstWordsPerLayer * int64_t(count))
    return fail(HICACHE_EINVAL, "opts.burst_words holds " + std::to_string(o.burst_words_len) +
                                    " words; the burst needs " +
                                    std::to_string(kBurstWordsPerLayer) + " per layer (" +
                                    std::to_string(kBurstWordsPerLayer * int64_t(count)) + ")");
  if (reinterpret_cast<uintptr_t>(o.burst_words) % 4 != 0)
    return fail(HICACHE_EALIGN, "opts.burst_words is not 4-byte aligned");
  return HICACHE_OK;
}

LaunchCfg launch_cfg(const hicache_opts& o) { return LaunchCfg{o.max_ctas, o.device_error}; }

hicache_path resolve_path(const Prepared& pr, Dir dir, int32_t layers) {
  if (pr.o.path != HICACHE_PATH_AUTO) return static_cast<hicache_path>(pr.o.path);
  return choose_path(pr.pools, pr.o, pr.idx, dir, layers);
}

void record_events(cudaEvent_t* evs, int32_t count, cudaStream_t stream) {
  if (!evs) return;
  for (int32_t i = 0; i < count; ++i)
    if (evs[i]) cudaEventRecord(evs[i], stream);
}

hicache_status load_layers(const Prepared& pr, int32_t layer_begin, int32_t layer_end,
                           cudaStream_t stream, cudaEvent_t* evs) {
  const int32_t count = layer_end - layer_begin;
  const hicache_path path = resolve_path(pr, kPagedToDev, count);
  if (path == HICACHE_PATH_STAGED)
    return staged_load(pr.pools, pr.o, pr.idx, layer_begin, layer_end, stream, evs);
  const SideSpec side = host_side(pr.pools);
  // one layer is one launch and its event either way: the signalling burst
  // would only add its stream hand-offs
  if (pr.o.burst_words && count > 1 && signaled_burst_available())
    return signaled_burst(pr.pools, side, pr.idx, pr.o, layer_begin, layer_end, stream, evs);
  const LaunchCfg cfg = launch_cfg(pr.o);
  for (int32_t l = layer_begin; l < layer_end; ++l) {
    hicache_status st = launch_rows(pr.pools, side, pr.idx.dev_gpu, pr.idx.host_gpu, pr.idx.bits,
                                    0, pr.idx.n, kPagedToDev, l, l + 1, cfg, stream);
    if (st != HICACHE_OK) {
      record_events(evs ? evs + (l - layer_begin) : nullptr, count - (l - layer_begin), stream);
      return st;
    }
    if (evs && evs[l - layer_begin]) {
      const cudaError_t e = cudaEventRecord(evs[l - layer_begin], stream);
      if (e != cudaSuccess) {
        st = cuda_fail(e, "cudaEventRecord(layer_done)");
        record_events(evs + (l - layer_begin) + 1, count - (l - layer_begin) - 1, stream);
        return st;
      }
    }
  }
  return HICACHE_OK;
}

}  // namespace
}  // namespace hk

using namespace hk;

extern "C" hicache_status hicache_backup_all_layers(const hicache_pool* pools, int32_t num_pools,
                                                    const void* device_indices,
                                                    const void* host_indices, int32_t index_bits,
                                                    int64_t n, const hicache_opts* opts,
                                                    cudaStream_t stream) {
  clear_error();
  Prepared pr;
  hicache_status st = prepare(pools, num_pools, device_indices, host_indices, index_bits, n, opts,
                              /*dest_is_device=*/false, false, 0, 0, &pr);
  if (st != HICACHE_OK || n == 0) return st;
  st = stage_indices(&pr, stream);
  if (st != HICACHE_OK) return st;
  const hicache_path path = resolve_path(pr, kDevToPaged, pr.pools[0].L);
  if (path == HICACHE_PATH_STAGED)
    return staged_backup(pr.pools, pr.o, pr.idx, stream);
  return launch_rows(pr.pools, host_side(pr.pools), pr.idx.dev_gpu, pr.idx.host_gpu, pr.idx.bits,
                     0, pr.idx.n, kDevToPaged, 0, pr.pools[0].L, launch_cfg(pr.o), stream);
}

extern "C" hicache_status hicache_load_layer(const hicache_pool* pools, int32_t num_pools,
                                             int32_t layer, const void* host_indices,
                                             const void* device_indices, int32_t index_bits,
                                             int64_t n, const hicache_opts* opts,
                                             cudaStream_t stream, cudaEvent_t layer_done) {
  clear_error();
  cudaEvent_t evs[1] = {layer_done};
  Prepared pr;
  hicache_status st = prepare(pools, num_pools, device_indices, host_indices, index_bits, n, opts,
                              /*dest_is_device=*/true, true, layer, layer + 1, &pr);
  if (st == HICACHE_OK && n > 0) st = stage_indices(&pr, stream);
  if (st != HICACHE_OK || n == 0) {
    record_events(evs, 1, stream);
    return st;
  }
  return load_layers(pr, layer, layer + 1, stream, evs);
}

extern "C" hicache_status hicache_load_burst(const hicache_pool* pools, int32_t num_pools,
                                             int32_t layer_begin, int32_t layer_end,
                                             const void* host_indices, const void* device_indices,
                                             int32_t index_bits, int64_t n,
                                             const hicache_opts* opts, cudaStream_t stream,
                                             cudaEvent_t* layer_done) {
  clear_error();
  const int32_t count = layer_end > layer_begin ? layer_end - layer_begin : 0;
  Prepared pr;
  hicache_status st = prepare(pools, num_pools, device_indices, host_indices, index_bits, n, opts,
                              /*dest_is_device=*/true, true, layer_begin, layer_end, &pr);
  if (st == HICACHE_OK) st = check_burst_words(pr.o, count);
  if (st == HICACHE_OK && n > 0) st = stage_indices(&pr, stream);
  if (st != HICACHE_OK || n == 0) {
    record_events(layer_done, count, stream);
    return st;
  }
  return load_layers(pr, layer_begin, layer_end, stream, layer_done);
}

// ---------------------------------------------------------------------------
// Backup with library-owned staging memory, for callers that cannot allocate.
//
// The staging lives in a file-scope device array.  Host code must not use the
// array's name as a device address (in host code it names a host-side
// stand-in); the device address is resolved once per device with
// cudaGetSymbolAddress and handed to the staged backup as its two buffers.
//
// Everything that could place memory on the device is done by the set-up that
// opens every call, a call with no pairs included: resolving the address loads
// the module that holds the array (under CUDA's default lazy loading that is
// when the array is placed in HBM), the copy kernels the staged backup launches
// are loaded, and the calling thread's copy stream and events are created.
// After one such call on a device and thread, later calls take no device memory.

static __device__ __align__(256) unsigned char g_static_staging[HICACHE_STATIC_STAGING_BYTES];

namespace hk {
namespace {

std::mutex g_static_mu;
void* g_static_addr[64] = {};

// Device address of g_static_staging on the current device, resolved (and the
// staged backup's kernels loaded) once per device.  A cudaDeviceReset destroys
// the module and with it the cached address, so the entry point must not be
// used on a device after it was reset.
hicache_status static_staging_setup(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(HICACHE_EINVAL, "device ordinal above 63");
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_staging);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static staging array)");
      if (!p) return fail(HICACHE_ECUDA, "cudaGetSymbolAddress returned NULL for the staging array");
      const hicache_status st = load_staged_backup_kernels();
      if (st != HICACHE_OK) return st;
      g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
  }
  // the calling thread's copy stream and events (created once per thread)
  return staged_resources_ready();
}

}  // namespace
}  // namespace hk

extern "C" hicache_status hicache_backup_all_layers_static_staging(
    const hicache_pool* pools, int32_t num_pools, const void* device_indices,
    const void* host_indices, int32_t index_bits, int64_t n, const hicache_opts* opts,
    cudaStream_t stream) {
  clear_error();
  hicache_opts o = opts ? *opts : default_opts();
  // Pure host checks first, so that a rejected call touches no CUDA state.
  std::vector<PoolInfo> checked;
  hicache_status st = check_pools(pools, num_pools, &checked);
  if (st != HICACHE_OK) return st;
  constexpr int64_t kHalf = int64_t(HICACHE_STATIC_STAGING_BYTES) / 2;
  int64_t page_all_layers = 0;
  for (const PoolInfo& pi : checked)
    page_all_layers += int64_t(pi.T) * pi.L * pi.P * pi.token_bytes;
  if (page_all_layers > kHalf)
    return fail(HICACHE_ENOSTAGE, "one host page of all layers of all pools is " +
                                      std::to_string(page_all_layers) +
                                      " bytes, above the " + std::to_string(kHalf) +
                                      "-byte half of the static staging array");
  // The set-up runs before the empty-list return, so that a call with no
  // pairs serves as the warm-up that takes this entry point's device memory.
  void* base = nullptr;
  st = static_staging_setup(&base);
  if (st != HICACHE_OK) return st;
  o.path = HICACHE_PATH_STAGED;
  o.staging[0] = base;
  o.staging[1] = static_cast<unsigned char*>(base) + kHalf;
  o.staging_bytes = size_t(kHalf);
  Prepared pr;
  st = prepare(pools, num_pools, device_indices, host_indices, index_bits, n, &o,
               /*dest_is_device=*/false, false, 0, 0, &pr);
  if (st != HICACHE_OK || n == 0) return st;
  return staged_backup(pr.pools, pr.o, pr.idx, stream);
}

extern "C" hicache_status hicache_auto_path(const hicache_pool* pools, int32_t num_pools,
                                            const void* device_indices, const void* host_indices,
                                            int32_t index_bits, int64_t n,
                                            const hicache_opts* opts, int32_t op, int32_t layers,
                                            int32_t* path_out) {
  clear_error();
  if (!path_out) return fail(HICACHE_EINVAL, "path_out is NULL");
  if (op != HICACHE_OP_BACKUP && op != HICACHE_OP_LOAD)
    return fail(HICACHE_EINVAL, "op must be HICACHE_OP_BACKUP or HICACHE_OP_LOAD");
  std::vector<PoolInfo> checked;
  hicache_status st = check_pools(pools, num_pools, &checked);
  if (st != HICACHE_OK) return st;
  const hicache_opts o = opts ? *opts : default_opts();
  st = check_opts(o);
  if (st == HICACHE_OK) st = check_index_args(device_indices, host_indices, index_bits, n);
  if (st != HICACHE_OK) return st;
  if (o.path != HICACHE_PATH_AUTO) {
    *path_out = o.path;
    return HICACHE_OK;
  }
  IndexSet idx;
  idx.bits = index_bits;
  idx.n = n;
  if (o.index_location == HICACHE_INDEX_HOST) {
    idx.dev_cpu = device_indices;
    idx.host_cpu = host_indices;
  }
  *path_out = choose_path(checked, o, idx, op == HICACHE_OP_BACKUP ? kDevToPaged : kPagedToDev,
                          op == HICACHE_OP_BACKUP ? checked[0].L : layers);
  return HICACHE_OK;
}

extern "C" hicache_status hicache_plan_runs(const void* device_indices, const void* host_indices,
                                            int32_t index_bits, int64_t n, int32_t page_size,
                                            hicache_run* runs_out, int64_t runs_cap,
                                            int64_t* num_runs, int64_t* full_pages) {
  clear_error();
  hicache_status st = check_index_args(device_indices, host_indices, index_bits, n);
  if (st != HICACHE_OK) return st;
  return plan_runs(device_indices, host_indices, index_bits, n, page_size, runs_out, runs_cap,
                   num_runs, full_pages);
}

extern "C" hicache_status hicache_check_pairs(const hicache_pool* pools, int32_t num_pools,
                                              const void* device_indices, const void* host_indices,
                                              int32_t index_bits, int64_t n,
                                              int32_t dest_is_device) {
  clear_error();
  std::vector<PoolInfo> checked;
  hicache_status st = check_pools(pools, num_pools, &checked);
  if (st != HICACHE_OK) return st;
  if (dest_is_device != 0 && dest_is_device != 1)
    return fail(HICACHE_EINVAL, "dest_is_device must be 0 or 1");
  st = check_index_args(device_indices, host_indices, index_bits, n);
  if (st != HICACHE_OK) return st;
  return check_pairs_host(checked, device_indices, host_indices, index_bits, n, dest_is_device == 1);
}

extern "C" hicache_status hicache_layer_checksum(const hicache_pool* pool, int32_t tensor,
                                                 int32_t layer, const void* device_indices,
                                                 int32_t index_bits, int64_t n, uint64_t* out_sum,
                                                 cudaStream_t stream) {
  clear_error();
  std::vector<PoolInfo> pools;
  hicache_status st = check_pools(pool, 1, &pools);
  if (st != HICACHE_OK) return st;
  st = check_index_args(device_indices, device_indices, index_bits, n);
  if (st != HICACHE_OK) return st;
  if (tensor < 0 || tensor >= pools[0].T) return fail(HICACHE_EINVAL, "tensor out of range");
  if (layer < 0 || layer >= pools[0].L) return fail(HICACHE_EINVAL, "layer out of range");
  if (!out_sum) return fail(HICACHE_EINVAL, "out_sum is NULL");
  if (n == 0) return HICACHE_OK;
  const void* v = nullptr;
  st = device_view(device_indices, Want::kDevice, "device_indices", &v);
  if (st != HICACHE_OK) return st;
  st = check_gpu_buffer(&out_sum, Want::kDevice, 8, "out_sum");
  if (st != HICACHE_OK) return st;
  return launch_checksum(pools[0], tensor, layer, v, index_bits, n, out_sum, stream);
}

extern "C" int64_t hicache_kernel_launches(void) { return kernel_launches(); }

extern "C" size_t hicache_index_staging_bytes(int64_t n, int32_t index_bits) {
  if (n <= 0 || (index_bits != 32 && index_bits != 64)) return 0;
  return 2 * index_array_bytes(n, index_bits);
}

extern "C" const char* hicache_last_error(void) { return last_error().c_str(); }

extern "C" int32_t hicache_abi_version(void) { return HICACHE_ABI_VERSION; }
