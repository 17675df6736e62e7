/*
 * hicache_oracle.h -- reference CPU implementation of the paged KV-cache
 * transfer (HiCache all-layer backup and per-layer load-back).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no header, helper or constant with the CUDA
 * path.
 *
 * Semantics followed:
 *   - "[HiCache] Support hybrid-pool staged write-back JIT kernel" (sglang PR
 *     #28434 summary), section "key source excerpts", the CPU simulation of the
 *     staged lf->pf copy: for every layer, the host rows named by the
 *     destination indices receive the device rows named by the source indices
 *     of that layer.
 *   - The host pool is page-first: one host page holds, for every layer in
 *     order, page_size token rows ("[HiCache] Run the host->device load-back
 *     enqueue on a loader thread", Motivation: the page_first_direct layout).
 *     A token row of one tensor is row_bytes bytes, so host token h of layer l
 *     starts at byte ((h / page_size) * num_layers + l) * page_size * row_bytes
 *     + (h % page_size) * row_bytes.
 *   - The device pool is layer-first: one buffer per layer, slot d of layer l
 *     starting at byte d * row_bytes of that layer's buffer.
 *   - Load-back of layer l is the inverse copy for that layer alone ("Run the
 *     host->device load-back enqueue on a loader thread", Motivation: the
 *     per-layer load_to_device_per_layer).
 *
 * All data are opaque bytes; there is no arithmetic on values.  Indices are
 * int64 token indices (a caller holding int32 indices widens them first, which
 * is exact).  Parity pins: see the oracle tests (hand-written golden images,
 * the numpy-shape restatement, round trip, untouched bytes, layout-structure
 * invariants and planted-mutation controls).
 */
#ifndef HICACHE_ORACLE_H
#define HICACHE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of the oracle functions. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_OUT_OF_RANGE (-2)

/*
 * All-layer backup (device -> host) of one tensor of one pool.
 *   device_layers : num_layers pointers, device_layers[l] = image of layer l,
 *                   device_slots * row_bytes bytes each.
 *   host          : image of the page-first host tensor,
 *                   host_pages * num_layers * page_size * row_bytes bytes.
 *   device_idx[i] -> host_idx[i], i < n.
 * Every host row named by a pair receives, for every layer, the device row of
 * that layer named by the same pair; every other host byte is left unchanged.
 */
int oracle_backup_all_layers(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                             int64_t device_slots, int64_t host_pages,
                             const uint8_t* const* device_layers, uint8_t* host,
                             const int64_t* device_idx, const int64_t* host_idx, int64_t n);

/*
 * Load-back of one layer (host -> device) of one tensor of one pool.
 *   device_layer  : image of layer `layer`, device_slots * row_bytes bytes.
 *   host          : image of the page-first host tensor.
 *   host_idx[i] -> device_idx[i], i < n.
 * Every device row named by a pair receives the host row of layer `layer`
 * named by the same pair; every other device byte is left unchanged.
 */
int oracle_load_layer(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                      int64_t device_slots, int64_t host_pages, int64_t layer,
                      uint8_t* device_layer, const uint8_t* host,
                      const int64_t* host_idx, const int64_t* device_idx, int64_t n);

/*
 * Load-back of layers [layer_begin, layer_end) in increasing order, one
 * oracle_load_layer call per layer.
 *   device_layers : num_layers pointers as in oracle_backup_all_layers.
 */
int oracle_load_burst(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                      int64_t device_slots, int64_t host_pages,
                      int64_t layer_begin, int64_t layer_end,
                      uint8_t* const* device_layers, const uint8_t* host,
                      const int64_t* host_idx, const int64_t* device_idx, int64_t n);

/*
 * The page_first host layout: token-major, [host token][layer][row].  It is the
 * shape of the staging buffer in "[HiCache] Support hybrid-pool staged
 * write-back JIT kernel" (sglang PR #28434 summary), key source excerpts
 * (staging_token_capacity x layer_num x element_dim), on which the CPU
 * simulation writes dst[dst_indices, layer] = src[src_indices].  Host token h
 * of layer l starts at byte (h * num_layers + l) * row_bytes; pages play no
 * part in the addressing (a page is page_size consecutive tokens).
 *   host_tokens : tokens of the host tensor (host_pages * page_size).
 */
int oracle_pf_backup_all_layers(int64_t num_layers, int64_t row_bytes, int64_t device_slots,
                                int64_t host_tokens, const uint8_t* const* device_layers,
                                uint8_t* host, const int64_t* device_idx, const int64_t* host_idx,
                                int64_t n);

int oracle_pf_load_layer(int64_t num_layers, int64_t row_bytes, int64_t device_slots,
                         int64_t host_tokens, int64_t layer, uint8_t* device_layer,
                         const uint8_t* host, const int64_t* host_idx, const int64_t* device_idx,
                         int64_t n);

#ifdef __cplusplus
}
#endif
#endif /* HICACHE_ORACLE_H */
