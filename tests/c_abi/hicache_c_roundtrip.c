/*
 * hicache_c_roundtrip.c -- the C ABI used from plain C99, with no Python.
 *
 * Test program: allocates a small MHA pool with the CUDA runtime (device layers
 * with cudaMalloc, the page-first host pool with cudaHostAlloc), backs up a
 * list of whole pages with hicache_backup_all_layers, loads them back into
 * other device pages with a single-launch hicache_load_burst, repeats both on
 * the staged path with cudaMalloc'd staging buffers, backs up once more with
 * the allocation-free entry point, and checks every byte of both pools against
 * the CPU oracle (test infrastructure, linked only by tests).  It also asks
 * hicache_auto_path for the path.  Exit status 0 means bit-exact; it prints the
 * first mismatch otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "hicache.h"
#include "hicache_oracle.h"

#define L 3
#define T 2
#define HEADS 2
#define DIM 64
#define ESIZE 2
#define R (HEADS * DIM * ESIZE)
#define P 16
#define SLOTS 1024
#define HPAGES 64
#define NPAGES 10

#define CHECK_CUDA(x)                                                         \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x,               \
              cudaGetErrorString(e_));                                        \
      return 2;                                                               \
    }                                                                         \
  } while (0)

#define CHECK_HK(x)                                                           \
  do {                                                                        \
    hicache_status s_ = (x);                                                  \
    if (s_ != HICACHE_OK) {                                                   \
      fprintf(stderr, "%s:%d %s: status %d: %s\n", __FILE__, __LINE__, #x,    \
              (int)s_, hicache_last_error());                                 \
      return 3;                                                               \
    }                                                                         \
  } while (0)

static uint32_t lcg(uint32_t* s) {
  *s = *s * 1664525u + 1013904223u;
  return *s >> 8;
}

/* n distinct values below `total`, seeded (Fisher-Yates over a scratch array). */
static void sample(uint32_t seed, int64_t total, int64_t n, const int64_t* avoid, int64_t navoid,
                   int64_t* out) {
  int64_t* all = (int64_t*)malloc(sizeof(int64_t) * (size_t)total);
  int64_t m = 0;
  for (int64_t v = 0; v < total; ++v) {
    int skip = 0;
    for (int64_t k = 0; k < navoid; ++k) skip |= (avoid[k] == v);
    if (!skip) all[m++] = v;
  }
  for (int64_t i = 0; i < n; ++i) {
    int64_t j = i + (int64_t)(lcg(&seed) % (uint32_t)(m - i));
    int64_t t = all[i];
    all[i] = all[j];
    all[j] = t;
    out[i] = all[i];
  }
  free(all);
}

int main(void) {
  const size_t layer_bytes = (size_t)SLOTS * R;
  const size_t host_bytes = (size_t)HPAGES * L * P * R;
  const int64_t n = (int64_t)NPAGES * P;
  uint32_t seed = 12345;

  /* pools */
  void* dev[T * L];
  uint8_t* dev_img[T * L];
  uint8_t* host[T];
  uint8_t* host_img[T];
  for (int i = 0; i < T * L; ++i) {
    CHECK_CUDA(cudaMalloc(&dev[i], layer_bytes));
    dev_img[i] = (uint8_t*)malloc(layer_bytes);
    for (size_t b = 0; b < layer_bytes; ++b) dev_img[i][b] = (uint8_t)lcg(&seed);
    CHECK_CUDA(cudaMemcpy(dev[i], dev_img[i], layer_bytes, cudaMemcpyHostToDevice));
  }
  for (int t = 0; t < T; ++t) {
    CHECK_CUDA(cudaHostAlloc((void**)&host[t], host_bytes, cudaHostAllocDefault));
    host_img[t] = (uint8_t*)malloc(host_bytes);
    for (size_t b = 0; b < host_bytes; ++b) host[t][b] = host_img[t][b] = (uint8_t)(b * 7 + t);
  }
  hicache_pool pool;
  memset(&pool, 0, sizeof(pool));
  pool.num_layers = L;
  pool.num_tensors = T;
  pool.head_num = HEADS;
  pool.head_dim = DIM;
  pool.dtype_size = ESIZE;
  pool.page_size = P;
  pool.page_granular = 0;
  pool.layout = HICACHE_LAYOUT_PAGE_FIRST_DIRECT;
  pool.device_slots = SLOTS;
  pool.host_pages = HPAGES;
  pool.device_layers = dev;
  pool.host_tensors = (void* const*)host;

  /* pairs: NPAGES random device pages -> NPAGES random host pages, in pinned memory */
  int64_t dpages[NPAGES], hpages[NPAGES], dpages2[NPAGES];
  sample(7, SLOTS / P, NPAGES, NULL, 0, dpages);
  sample(8, HPAGES, NPAGES, NULL, 0, hpages);
  sample(9, SLOTS / P, NPAGES, dpages, NPAGES, dpages2);
  int64_t *d_idx, *h_idx, *d2_idx;
  CHECK_CUDA(cudaHostAlloc((void**)&d_idx, sizeof(int64_t) * (size_t)n, cudaHostAllocDefault));
  CHECK_CUDA(cudaHostAlloc((void**)&h_idx, sizeof(int64_t) * (size_t)n, cudaHostAllocDefault));
  CHECK_CUDA(cudaHostAlloc((void**)&d2_idx, sizeof(int64_t) * (size_t)n, cudaHostAllocDefault));
  for (int64_t k = 0; k < NPAGES; ++k)
    for (int64_t t = 0; t < P; ++t) {
      d_idx[k * P + t] = dpages[k] * P + t;
      h_idx[k * P + t] = hpages[k] * P + t;
      d2_idx[k * P + t] = dpages2[k] * P + t;
    }

  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
  hicache_opts opts;
  memset(&opts, 0, sizeof(opts));
  opts.path = HICACHE_PATH_AUTO;
  opts.index_location = HICACHE_INDEX_HOST;

  /* backup, then check the host pool against the oracle */
  CHECK_HK(hicache_backup_all_layers(&pool, 1, d_idx, h_idx, 64, n, &opts, stream));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  for (int t = 0; t < T; ++t) {
    const uint8_t* layers[L];
    for (int l = 0; l < L; ++l) layers[l] = dev_img[t * L + l];
    if (oracle_backup_all_layers(L, P, R, SLOTS, HPAGES, layers, host_img[t], d_idx, h_idx, n) != 0)
      return 4;
    for (size_t b = 0; b < host_bytes; ++b)
      if (host[t][b] != host_img[t][b]) {
        fprintf(stderr, "backup: tensor %d byte %zu differs\n", t, b);
        return 1;
      }
  }

  /* single-launch burst with one event per layer, then check the device pool */
  uint32_t* words;
  CHECK_CUDA(cudaMalloc((void**)&words, sizeof(uint32_t) * 4 * L));
  opts.burst_words = words;
  opts.burst_words_len = 4 * L;
  cudaEvent_t ev[L];
  for (int l = 0; l < L; ++l) CHECK_CUDA(cudaEventCreateWithFlags(&ev[l], cudaEventDisableTiming));
  CHECK_HK(hicache_load_burst(&pool, 1, 0, L, h_idx, d2_idx, 64, n, &opts, stream, ev));
  for (int l = 0; l < L; ++l) CHECK_CUDA(cudaEventSynchronize(ev[l]));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  uint8_t* got = (uint8_t*)malloc(layer_bytes);
  for (int t = 0; t < T; ++t) {
    uint8_t* layers[L];
    for (int l = 0; l < L; ++l) layers[l] = dev_img[t * L + l];
    if (oracle_load_burst(L, P, R, SLOTS, HPAGES, 0, L, layers, host_img[t], h_idx, d2_idx, n) != 0)
      return 4;
    for (int l = 0; l < L; ++l) {
      CHECK_CUDA(cudaMemcpy(got, dev[t * L + l], layer_bytes, cudaMemcpyDeviceToHost));
      for (size_t b = 0; b < layer_bytes; ++b)
        if (got[b] != dev_img[t * L + l][b]) {
          fprintf(stderr, "burst: tensor %d layer %d byte %zu differs\n", t, l, b);
          return 1;
        }
    }
  }
  /* a rejected call still completes the events: duplicate device destination */
  d2_idx[1] = d2_idx[0];
  if (hicache_load_burst(&pool, 1, 0, L, h_idx, d2_idx, 64, n, &opts, stream, ev) != HICACHE_EDUP)
    return 5;
  for (int l = 0; l < L; ++l) CHECK_CUDA(cudaEventSynchronize(ev[l]));

  /* the staged path: backup to other host pages, then a burst into other
     device pages.  The staging holds 7 host pages of all layers: the backup
     copies 8 of its 10 pages through it (chunks of 7 + 1) and the last 2
     zero-copy.  The load reads layer 0 zero-copy and copies layers 1-2 as one
     group (10 pages of two layers fit in one chunk). */
  int64_t hpages3[NPAGES], dpages3[NPAGES];
  sample(10, HPAGES, NPAGES, hpages, NPAGES, hpages3);
  sample(11, SLOTS / P, NPAGES, dpages, NPAGES, dpages3);
  for (int64_t k = 0; k < NPAGES; ++k)
    for (int64_t t = 0; t < P; ++t) {
      h_idx[k * P + t] = hpages3[k] * P + t;
      d2_idx[k * P + t] = dpages3[k] * P + t;
    }
  const size_t stage_bytes = (size_t)7 * T * L * P * R;
  void* staging[2];
  for (int b = 0; b < 2; ++b) CHECK_CUDA(cudaMalloc(&staging[b], stage_bytes));
  hicache_opts sopts;
  memset(&sopts, 0, sizeof(sopts));
  sopts.path = HICACHE_PATH_STAGED;
  sopts.index_location = HICACHE_INDEX_HOST;
  sopts.staging[0] = staging[0];
  sopts.staging[1] = staging[1];
  sopts.staging_bytes = stage_bytes;
  CHECK_HK(hicache_backup_all_layers(&pool, 1, d_idx, h_idx, 64, n, &sopts, stream));
  CHECK_HK(hicache_load_burst(&pool, 1, 0, L, h_idx, d2_idx, 64, n, &sopts, stream, ev));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  for (int t = 0; t < T; ++t) {
    uint8_t* layers[L];
    for (int l = 0; l < L; ++l) layers[l] = dev_img[t * L + l];
    if (oracle_backup_all_layers(L, P, R, SLOTS, HPAGES, (const uint8_t* const*)layers,
                                 host_img[t], d_idx, h_idx, n) != 0)
      return 4;
    if (oracle_load_burst(L, P, R, SLOTS, HPAGES, 0, L, layers, host_img[t], h_idx, d2_idx, n) != 0)
      return 4;
    for (size_t b = 0; b < host_bytes; ++b)
      if (host[t][b] != host_img[t][b]) {
        fprintf(stderr, "staged backup: tensor %d byte %zu differs\n", t, b);
        return 1;
      }
    for (int l = 0; l < L; ++l) {
      CHECK_CUDA(cudaMemcpy(got, dev[t * L + l], layer_bytes, cudaMemcpyDeviceToHost));
      for (size_t b = 0; b < layer_bytes; ++b)
        if (got[b] != dev_img[t * L + l][b]) {
          fprintf(stderr, "staged burst: tensor %d layer %d byte %zu differs\n", t, l, b);
          return 1;
        }
    }
  }

  /* the allocation-free backup, as a C caller with no device allocator of its
     own would use it: one call with no pairs first (the set-up that takes the
     library's static staging array), then the pairs, to yet other host pages */
  int64_t hpages4[NPAGES], used[2 * NPAGES];
  for (int64_t k = 0; k < NPAGES; ++k) {
    used[k] = hpages[k];
    used[NPAGES + k] = hpages3[k];
  }
  sample(12, HPAGES, NPAGES, used, 2 * NPAGES, hpages4);
  for (int64_t k = 0; k < NPAGES; ++k)
    for (int64_t t = 0; t < P; ++t) h_idx[k * P + t] = hpages4[k] * P + t;
  CHECK_HK(hicache_backup_all_layers_static_staging(&pool, 1, NULL, NULL, 64, 0, NULL, stream));
  CHECK_HK(hicache_backup_all_layers_static_staging(&pool, 1, d_idx, h_idx, 64, n, NULL, stream));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  for (int t = 0; t < T; ++t) {
    const uint8_t* layers[L];
    for (int l = 0; l < L; ++l) layers[l] = dev_img[t * L + l];
    if (oracle_backup_all_layers(L, P, R, SLOTS, HPAGES, layers, host_img[t], d_idx, h_idx, n) != 0)
      return 4;
    for (size_t b = 0; b < host_bytes; ++b)
      if (host[t][b] != host_img[t][b]) {
        fprintf(stderr, "static-staging backup: tensor %d byte %zu differs\n", t, b);
        return 1;
      }
  }

  /* AUTO's rule from C: with a small CTA budget and staging the rule still
     says zero-copy here, because these host pages (12 KiB) are far below the
     1 MiB a staged DMA needs; without a budget it is zero-copy too */
  int32_t path = -1;
  sopts.path = HICACHE_PATH_AUTO;
  sopts.max_ctas = 8;
  CHECK_HK(hicache_auto_path(&pool, 1, d_idx, h_idx, 64, n, &sopts, HICACHE_OP_BACKUP, 0, &path));
  if (path != HICACHE_PATH_ZERO_COPY) return 6;
  CHECK_HK(hicache_auto_path(&pool, 1, d_idx, h_idx, 64, n, NULL, HICACHE_OP_LOAD, L, &path));
  if (path != HICACHE_PATH_ZERO_COPY) return 6;

  printf("c abi round trip ok: %d layers, %d tensors, %d pages, launches %lld\n", L, T, NPAGES,
         (long long)hicache_kernel_launches());
  return 0;
}
