/*
 * hicache.h -- C ABI of the GB300 paged KV-cache transfer library.
 *
 * The library moves token rows between a layer-first device KV pool (HBM) and
 * a page-first pinned host pool, driven by lists of (device slot, host slot)
 * pairs.  Two operations exist:
 *
 *   - the all-layer backup (device -> host write-back), and
 *   - the per-layer load-back (host -> device), one layer per call or a burst
 *     of layers with one completion event per layer, so that a consumer can
 *     start on layer l while layer l+1 is still being copied.
 *
 * Passages that define the operations:
 *   - "[HiCache] Support hybrid-pool staged write-back JIT kernel" (sglang PR
 *     #28434 summary), key source excerpts: backup_from_device_all_layer of the
 *     MHA host pool and the CPU simulation of the staged lf->pf copy (for every
 *     layer, the host rows named by the destination indices take the device rows
 *     named by the source indices).
 *   - "[HiCache] Run the host->device load-back enqueue on a loader thread"
 *     (sglang PR #38472), Motivation: per-layer load_to_device_per_layer with the
 *     page_first_direct host layout and LayerDoneCounter.wait_until in the
 *     attention layers; Modifications: a failed load still completes every layer
 *     event so that a waiting consumer cannot hang.
 *
 * Layouts (all data are opaque bytes; no arithmetic is done on values):
 *   R = head_num * head_dim * dtype_size bytes per token row of one tensor.
 *   Device: tensor t, layer l is one buffer of device_slots rows; slot d starts
 *           at byte d * R of device_layers[t * num_layers + l].
 *   Host:   tensor t is one buffer, page-first: host token h of layer l starts at
 *           byte ((h / P) * num_layers + l) * P * R + (h % P) * R of
 *           host_tensors[t].  One (page, layer) block is P * R contiguous bytes
 *           and one page holds the blocks of all layers in layer order.
 *   That host order is HICACHE_LAYOUT_PAGE_FIRST_DIRECT (the default).  With
 *   HICACHE_LAYOUT_PAGE_FIRST the host tensor is token-major instead, the shape
 *   (token, layer, element) of the staging buffer in the sglang PR #28434
 *   summary: host token h of layer l starts at byte (h * num_layers + l) * R.
 *   Either way one host page (all layers) is P * num_layers * R contiguous bytes.
 *   A page-granular pool (DSA indexer-K: 128 fp8 values + one 4-byte scale per
 *   token) uses the same formulas; it only requires that the pairs cover whole,
 *   page-aligned pages, so that with the direct layout the library may move one
 *   P * R page row at a time even when R is not a multiple of 16.
 *
 * Ownership and ordering:
 *   The caller owns every pool, index array, staging buffer, stream and event;
 *   the library allocates no device or pinned memory on any call.  All work is
 *   stream-ordered on `stream`: it starts after everything enqueued on `stream`
 *   before the call (so device indices written there are read safely) and ends
 *   before anything enqueued on `stream` after the call returns.  Index arrays,
 *   pools and staging buffers must stay valid until `stream` has passed the
 *   call.  Calls that share a staging buffer must be ordered by the caller.
 *   On first use on a thread and device, the single-launch burst creates one
 *   library stream and the staged path two (copy engine and zero-copy share),
 *   with a few events, kept until the process exits; bursts issued from one
 *   thread share that stream, so their layer events are recorded in issue
 *   order.
 *
 * Errors:
 *   Every function returns a hicache_status and never aborts or throws across
 *   the ABI.  hicache_last_error() returns a per-thread message for the last
 *   non-OK status.  Argument and index validation complete before any copy is
 *   enqueued, so a rejected call moves no byte.  A load call that fails still
 *   records every layer-done event it was given on `stream`.  Buffers the GPU
 *   writes (pool tensors, staging, opts.device_error, opts.burst_words,
 *   opts.index_staging) are checked for alignment (HICACHE_EALIGN) and, except
 *   the per-layer device pointers, for the kind of memory (HICACHE_EINVAL).
 */
#ifndef HICACHE_H
#define HICACHE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HICACHE_ABI_VERSION 5 /* 5: adds hicache_auto_path; 4: adds hicache_check_pairs */

typedef enum hicache_status {
  HICACHE_OK = 0,
  HICACHE_EINVAL = 1,   /* bad argument: null pointer, bad shape, layer range, pool mismatch,
                           pool memory the GPU cannot address, page-granular pairs that are not
                           whole aligned pages */
  HICACHE_ERANGE = 2,   /* an index is negative or beyond its pool */
  HICACHE_EDUP = 3,     /* two pairs name the same destination row */
  HICACHE_EALIGN = 4,   /* row bytes not a multiple of 4, or a base pointer not 4-byte aligned */
  HICACHE_ECUDA = 5,    /* a CUDA runtime call failed; hicache_last_error() names it */
  HICACHE_ENOSTAGE = 6  /* the staged path was requested without usable staging buffers */
} hicache_status;

typedef enum hicache_path {
  HICACHE_PATH_AUTO = 0,      /* the library chooses per call (hicache_auto_path gives the rule) */
  HICACHE_PATH_ZERO_COPY = 1, /* SMs read and write the mapped pinned host pool directly */
  HICACHE_PATH_STAGED = 2     /* gather/scatter through HBM staging + copy-engine DMA */
} hicache_path;

typedef enum hicache_index_location {
  /* Both index arrays are in pinned (page-locked) host memory: the CPU validates
   * them completely before enqueueing (range, duplicate destinations, whole
   * pages) and the GPU reads them through their mapping (or from
   * opts->index_staging).  Device memory passed here is rejected with
   * HICACHE_EINVAL before the CPU reads it.  The check of distinct
   * destinations keeps a bitmap of one bit per destination row on each calling
   * thread, reused by later calls (for a destination space above 2^28 rows that
   * a list uses sparsely, a sorted copy of the list instead). */
  HICACHE_INDEX_HOST = 0,
  /* Both index arrays are in device memory and may still be being written on
   * `stream`.  The CPU does not read them: kernels skip pairs that are out of
   * range (or, for a page-granular pool, not page-aligned) and OR an error bit
   * into opts->device_error when given.  Distinct destinations, and for a
   * page-granular pool in the page_first_direct layout whole pages, are the
   * caller's responsibility in this mode: such a pool moves one page row per
   * page_size pairs, addressed by the first pair of the group alone (the
   * others are not read), so a bad first pair skips the whole page. */
  HICACHE_INDEX_DEVICE = 1
} hicache_index_location;

typedef enum hicache_layout {
  HICACHE_LAYOUT_PAGE_FIRST_DIRECT = 0, /* host [page][layer][token][row] */
  HICACHE_LAYOUT_PAGE_FIRST = 1         /* host [token][layer][row] (pages of P tokens) */
} hicache_layout;

/* Bits kernels OR into hicache_opts.device_error. */
#define HICACHE_DEVERR_RANGE 1u     /* a pair was out of range and skipped */
#define HICACHE_DEVERR_PAGE_ALIGN 2u /* a page-granular pair was not page-aligned and skipped */
#define HICACHE_DEVERR_TIMEOUT 4u    /* a bulk copy of the staged path did not land within one
                                        second; that launch stopped early (never expected) */

typedef struct hicache_pool {
  int32_t num_layers;     /* L: layers of this pool */
  int32_t num_tensors;    /* T: 2 = MHA K and V, 1 = MLA latent or DSA indexer */
  int32_t head_num;       /* KV heads per token row (1 for MLA latent and indexer) */
  int32_t head_dim;       /* elements per head (576 for MLA latent, 132 for the indexer) */
  int32_t dtype_size;     /* bytes per element (2 for bf16, 1 for uint8/fp8) */
  int32_t page_size;      /* P: tokens per page, the same for device and host */
  int32_t page_granular;  /* 1: pairs must cover whole page-aligned pages (DSA indexer) */
  int32_t layout;         /* hicache_layout of the host tensors */
  int64_t device_slots;   /* token rows per device layer buffer */
  int64_t host_pages;     /* pages of the host pool */
  void* const* device_layers; /* host array of T * L device pointers, [t * L + l] */
  void* const* host_tensors;  /* host array of T pinned host pointers (see layout) */
} hicache_pool;

typedef struct hicache_opts {
  int32_t path;            /* hicache_path */
  int32_t index_location;  /* hicache_index_location */
  int32_t max_ctas;        /* 0 = library default (for the host-link copies, one 256-thread CTA
                              per SM for a backup, one per two SMs for a load); else caps the
                              CTAs of each copy kernel, so that compute running at the same
                              time keeps the other SMs.  Copies of up to 76 CTAs against the
                              host pool take deep tasks (twice the bytes in flight per warp),
                              and a cap of 16 or fewer runs 512-thread CTAs (twice the warps).
                              Measured on GB300 beside a bf16 GEMM loop: 8 CTAs moved 123-158
                              GB/s, 16 CTAs 178-200, and cost the GEMM 5-19 % of its
                              throughput, against 20-32 % with one CTA per SM (backups between
                              about 18 and 26 CTAs move less than at 16 or 32).  A backup and
                              a load-back running at the same time moved the most together
                              with 76 on both calls (298-317 GB/s, against about 245 with the
                              defaults).  Below
                              HICACHE_AUTO_STAGED_BELOW_CTAS_* the AUTO path may switch to the
                              staged path (see hicache_auto_path). */
  int32_t reserved;        /* must be 0 */
  void* staging[2];        /* staged path: two device buffers used alternately, 16-byte aligned */
  size_t staging_bytes;    /* bytes of each staging buffer */
  cudaStream_t copy_stream;/* staged path: stream for the DMA copies (0 = library-internal) */
  uint32_t* device_error;  /* optional word in device or pinned host memory, 4-byte aligned;
                              kernels OR HICACHE_DEVERR_* bits into it */
  uint32_t* burst_words;   /* optional device memory of >= 4 words per burst layer: makes a
                              zero-copy hicache_load_burst one kernel launch for all its layers
                              (see hicache_load_burst); NULL = one launch per layer */
  int64_t burst_words_len; /* number of uint32 words at burst_words */
  void* index_staging;     /* optional device memory for host-located indices: after validating
                              them the call copies both arrays here (stream-ordered) and the kernels
                              read them from HBM instead of across the host link; needs
                              hicache_index_staging_bytes(n, index_bits) bytes, 16-byte aligned */
  size_t index_staging_bytes; /* bytes at index_staging */
} hicache_opts;

/*
 * All-layer backup (device -> host) of the pairs device_indices[i] ->
 * host_indices[i], i < n, for every layer and tensor of every pool.
 * Passage: sglang PR #28434 summary, key source excerpts
 * (backup_from_device_all_layer; CPU simulation of the staged lf->pf copy).
 *   pools, num_pools : 1..4 pools that share the pair list, the layer count and
 *                      the page size (e.g. MLA latent + DSA indexer-K).
 *   device_indices, host_indices : n token indices each, int32 or int64
 *                      (index_bits 32 or 64), located as opts->index_location.
 *   opts             : NULL for defaults (AUTO path, host-located indices).
 *   stream           : stream the work is ordered on.
 * Host destinations must be distinct (HICACHE_EDUP); sources may repeat.
 * Host bytes not named by a pair are never written.
 */
hicache_status hicache_backup_all_layers(const hicache_pool* pools, int32_t num_pools,
                                         const void* device_indices, const void* host_indices,
                                         int32_t index_bits, int64_t n,
                                         const hicache_opts* opts, cudaStream_t stream);

/*
 * Load-back (host -> device) of one layer: host_indices[i] -> device_indices[i]
 * for layer `layer` of every tensor of every pool.  If layer_done is not NULL
 * it is recorded on `stream` after the copies, also when the call fails.
 * Passage: sglang PR #38472, Motivation (per-layer load_to_device_per_layer)
 * and Modifications (every layer event completes on failure).
 * Device destinations must be distinct (HICACHE_EDUP); sources may repeat.
 */
hicache_status hicache_load_layer(const hicache_pool* pools, int32_t num_pools, int32_t layer,
                                  const void* host_indices, const void* device_indices,
                                  int32_t index_bits, int64_t n, const hicache_opts* opts,
                                  cudaStream_t stream, cudaEvent_t layer_done);

/*
 * Load-back burst: layers layer_begin .. layer_end-1 in increasing order; event
 * layer_done[l - layer_begin] completes once every pool's layer l has landed.
 * The indices are validated once for the whole burst.  layer_done holds
 * layer_end - layer_begin events (entries may be NULL).  On any failure every
 * non-NULL event is still recorded.
 * Passage: sglang PR #38472, Motivation (one burst of per-layer loads gated by
 * LayerDoneCounter.wait_until) and Modifications (failure completes every
 * layer event).
 * Without opts->burst_words, each layer is one kernel launch on `stream`
 * followed by cudaEventRecord(layer_done[...], stream).  With
 * opts->burst_words (device memory, at least 4 * (layer_end - layer_begin)
 * words, zeroed by the call itself), a zero-copy burst takes two launches when
 * a layer holds 16 MiB or more: the first layer alone (its event recorded on
 * `stream`), then one launch covering all other layers; a smaller burst is
 * that one launch alone.  Its tasks are handed out in layer order: the kernel
 * sets one word per group of layers once the group has landed, a library
 * stream forked from `stream` waits on each word with a stream memory wait and
 * records the group's layer events, and `stream` joins that stream before the
 * call returns.  A layer of 2 MiB or more (all pools) is a group of its own;
 * smaller layers form groups of about 2 MiB, whose events are recorded together
 * once the whole group has landed.  The words must not be shared by bursts that overlap on the
 * GPU.
 * The staged path reads the first layers of a burst of two or more layers
 * zero-copy on a library stream (the SMs read the host pool; one layer in
 * eight, at least one: the first with its own launch and event, the others
 * likewise, or, given opts->burst_words, as one signalling launch), then
 * copies groups of consecutive
 * layers of each host page per DMA, each group four times the previous (up to
 * about 4 MiB per copy, in chunks of pages that fit a staging buffer),
 * scatters each chunk in one launch, and records a group's events once its
 * last chunk has landed.  Its later layer events therefore arrive in groups,
 * each no earlier than its own layer's data.  The last quarter of the pages
 * of each group is read zero-copy on a library stream while the copy engine
 * moves the group's other pages, and so is a pool whose host page is under
 * 1 MiB beside a larger pool (one launch each per group); the group's events
 * also wait for that stream.  The staged backup likewise moves the last
 * quarter of its pages, and such small pools, zero-copy on a library stream
 * beside its DMAs.
 */
hicache_status hicache_load_burst(const hicache_pool* pools, int32_t num_pools,
                                  int32_t layer_begin, int32_t layer_end,
                                  const void* host_indices, const void* device_indices,
                                  int32_t index_bits, int64_t n, const hicache_opts* opts,
                                  cudaStream_t stream, cudaEvent_t* layer_done);

/* Bytes of the library's own device staging array used by
 * hicache_backup_all_layers_static_staging: two halves of 16 MiB. */
#define HICACHE_STATIC_STAGING_BYTES (32u << 20)

/*
 * All-layer backup through the staged path without any memory from the caller
 * or the CUDA allocator.  Same pairs, pools, result and errors as
 * hicache_backup_all_layers with HICACHE_PATH_STAGED, but the two staging
 * buffers are the halves of one device array of HICACHE_STATIC_STAGING_BYTES
 * that the library defines statically.  The pages have no counterpart for this
 * entry point: it exists for callers that cannot allocate device memory at
 * transfer time, such as a serving engine that reserved all free HBM for its KV
 * pool at start-up, or a thin C caller with no device allocator of its own.
 *   - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *     library routine.  opts->staging and opts->staging_bytes are ignored.
 *   - Warm-up: every call first makes sure, on the current device, that the
 *     module holding the array is loaded (under CUDA's default lazy module
 *     loading, that is when the array takes its 32 MiB of HBM), that the copy
 *     kernels this call launches are loaded, and that the calling thread's copy
 *     stream and events exist.  Only the first call on a device (and thread)
 *     does any of this.  A call with n = 0 does this set-up and nothing else,
 *     so a caller that is about to give the rest of HBM to its pools makes one
 *     such call first (per device, with that device current, and on each
 *     thread that will call it); later calls take no device memory.  Make that
 *     first call before any stream capture.  With CUDA_MODULE_LOADING=EAGER
 *     the array is placed in HBM when the library's module loads instead, and
 *     stays there until the process exits either way.
 *   - Do not call it on a device after cudaDeviceReset: the array's address
 *     is resolved once per device and would then be stale.
 *   - Host-located indices covering whole host pages are required, as for the
 *     staged path (HICACHE_EINVAL otherwise).
 *   - One host page of all layers of all pools must fit in one 16 MiB half;
 *     larger pages are rejected with HICACHE_ENOSTAGE and a message giving both
 *     sizes.  Any number of pages is handled, 16 MiB at a time.
 *   - Every call uses the same array.  Nothing in it needs to start at zero:
 *     each call writes every staging byte it copies out.  Calls that overlap on
 *     the GPU (for example on two streams without ordering) race on the array.
 */
hicache_status hicache_backup_all_layers_static_staging(const hicache_pool* pools,
                                                        int32_t num_pools,
                                                        const void* device_indices,
                                                        const void* host_indices,
                                                        int32_t index_bits, int64_t n,
                                                        const hicache_opts* opts,
                                                        cudaStream_t stream);

/* Operations, for hicache_auto_path. */
#define HICACHE_OP_BACKUP 0 /* hicache_backup_all_layers */
#define HICACHE_OP_LOAD 1   /* hicache_load_layer (1 layer) or hicache_load_burst */

/* Copy-CTA budgets (opts->max_ctas) below which HICACHE_PATH_AUTO takes the
 * staged path when it may (see hicache_auto_path), per direction. */
#define HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP 5
#define HICACHE_AUTO_STAGED_BELOW_CTAS_LOAD 5

/*
 * The path a call with opts->path == HICACHE_PATH_AUTO takes (host only; no
 * CUDA call, so a scheduler may ask ahead of the call).  Writes
 * HICACHE_PATH_ZERO_COPY or HICACHE_PATH_STAGED to *path_out.
 *   op     : HICACHE_OP_BACKUP or HICACHE_OP_LOAD.
 *   layers : for a load, the layers the call moves (1 for hicache_load_layer,
 *            layer_end - layer_begin for a burst); ignored for a backup.
 *   Index arrays are read only when opts->index_location is HICACHE_INDEX_HOST
 *   (then they must be host memory); n pairs of index_bits bits.
 * The rule, from measurements on GB300 beside a bf16 GEMM loop (zero-copy
 * bandwidth grows with its CTAs until about 16 of them fill the host link;
 * the staged path moves its bytes with the copy engine and needs SMs only for
 * short gather and scatter kernels, which pays off under a cap of 4 CTAs or
 * fewer):
 *   the staged path when all of these hold, else zero-copy:
 *   - opts->max_ctas is set (the caller keeps the other SMs for compute) and
 *     below HICACHE_AUTO_STAGED_BELOW_CTAS_BACKUP / _LOAD;
 *   - two staging buffers are given, holding at least one host page of every
 *     staged pool (of all layers for a backup, of one layer for a load);
 *   - host-located indices whose pairs are whole host pages;
 *   - the largest pool's host page (all layers of one tensor) is at least
 *     1 MiB, so that one DMA per page is not dominated by the copy engine's
 *     fixed cost per copy;
 *   - for a load, at least two layers (a single layer would be one small DMA
 *     per page).
 * Errors: the argument checks of the calls (pools, opts, index arguments),
 * HICACHE_EINVAL for a bad op or a NULL path_out.
 */
hicache_status hicache_auto_path(const hicache_pool* pools, int32_t num_pools,
                                 const void* device_indices, const void* host_indices,
                                 int32_t index_bits, int64_t n, const hicache_opts* opts,
                                 int32_t op, int32_t layers, int32_t* path_out);

/* Bytes of opts->index_staging that a call with n pairs of index_bits-bit
 * indices needs (both arrays, each 16-byte aligned). */
size_t hicache_index_staging_bytes(int64_t n, int32_t index_bits);

/* One maximal run of pairs: device slots d0.., host slots h0.., len pairs. */
typedef struct hicache_run {
  int64_t d0;
  int64_t h0;
  int64_t len;
} hicache_run;

/*
 * Run planner (host only; no CUDA call).  Splits n pairs in host memory into
 * maximal runs in which the device and the host slot both increase by one and
 * the host slot does not cross a page boundary.  Writes up to runs_cap runs and
 * stores the total count in *num_runs (runs_out may be NULL to count only) and,
 * if full_pages is not NULL, the number of runs that are one whole page-aligned
 * host page.  Replaces the per-chunk CPU copy descriptors that the per-layer
 * load builds (sglang PR #38472, Motivation).
 */
hicache_status hicache_plan_runs(const void* device_indices, const void* host_indices,
                                 int32_t index_bits, int64_t n, int32_t page_size,
                                 hicache_run* runs_out, int64_t runs_cap, int64_t* num_runs,
                                 int64_t* full_pages);

/*
 * Index validation alone (host only; no CUDA call): checks n pairs in host
 * memory against the pools exactly as a call with HICACHE_INDEX_HOST does
 * before it enqueues anything, and returns the status that call would return
 * for them.  In order of precedence:
 *   HICACHE_ERANGE - a device index outside [0, device_slots) or a host index
 *                    outside [0, host_pages * page_size) of some pool;
 *   HICACHE_EDUP   - a destination named twice: host slots when
 *                    dest_is_device is 0 (a backup), device slots when it is 1
 *                    (a load);
 *   HICACHE_EINVAL - for a page-granular pool, pairs that are not whole
 *                    page-aligned pages (n a multiple of page_size, every group
 *                    of page_size pairs one aligned page on both sides).
 * The pools are checked as by every call (HICACHE_EINVAL / HICACHE_EALIGN).
 * Lets a scheduler validate a pair list on its own thread, ahead of the call;
 * the cost is one pass over the runs of the list (about a nanosecond per pair
 * for lists of whole pages).
 * Passage: sglang PR #38472, Motivation (the per-layer CPU work this replaces).
 */
hicache_status hicache_check_pairs(const hicache_pool* pools, int32_t num_pools,
                                   const void* device_indices, const void* host_indices,
                                   int32_t index_bits, int64_t n, int32_t dest_is_device);

/*
 * Synthetic consumer (not a transfer): adds, over the pairs' device slots
 * device_indices[i], i < n, of layer `layer` of tensor `tensor` of `pool`, every
 * little-endian 32-bit word of each row into *out_sum (device memory, a uint64
 * the caller zeroes), modulo 2^64.  Used to show that a kernel gated by a
 * layer-done event sees that layer fully loaded.  R must be a multiple of 4;
 * indices must be device memory.  No counterpart in the pages: it stands in for
 * the attention layer that waits on the layer event.
 */
hicache_status hicache_layer_checksum(const hicache_pool* pool, int32_t tensor, int32_t layer,
                                      const void* device_indices, int32_t index_bits, int64_t n,
                                      uint64_t* out_sum, cudaStream_t stream);

/* Number of kernels this library has launched in this process (all threads and
 * devices).  Lets a caller count the GPU work a region of its program issued. */
int64_t hicache_kernel_launches(void);

/* Message for the last non-OK status returned on the calling thread. */
const char* hicache_last_error(void);

/* HICACHE_ABI_VERSION of the loaded library. */
int32_t hicache_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HICACHE_H */
