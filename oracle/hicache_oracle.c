/*
 * hicache_oracle.c -- plain, slow, obviously correct CPU loops for the paged
 * KV-cache transfer.  TEST INFRASTRUCTURE ONLY (see hicache_oracle.h for the
 * passages followed).  One memcpy per token row; no blocking, no run merging,
 * no reordering.
 */
#include "hicache_oracle.h"

#include <string.h>

/* Byte offset of host token h, layer l, in the page-first host tensor:
 * page h / page_size, then layer l inside that page, then token h % page_size
 * inside that (page, layer) block.  ("Run the host->device load-back enqueue on
 * a loader thread", Motivation: page_first_direct.) */
static int64_t host_row_offset(int64_t h, int64_t l, int64_t num_layers,
                               int64_t page_size, int64_t row_bytes) {
  int64_t page = h / page_size;
  int64_t token_in_page = h % page_size;
  int64_t block = page * num_layers + l;           /* (page, layer) block number */
  return block * page_size * row_bytes + token_in_page * row_bytes;
}

/* Byte offset of device slot d inside one layer-first device layer buffer. */
static int64_t device_row_offset(int64_t d, int64_t row_bytes) { return d * row_bytes; }

static int shape_ok(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                    int64_t device_slots, int64_t host_pages, int64_t n) {
  return num_layers > 0 && page_size > 0 && row_bytes > 0 && device_slots >= 0 &&
         host_pages >= 0 && n >= 0;
}

static int pairs_in_range(const int64_t* device_idx, const int64_t* host_idx, int64_t n,
                          int64_t device_slots, int64_t host_tokens) {
  for (int64_t i = 0; i < n; ++i) {
    if (device_idx[i] < 0 || device_idx[i] >= device_slots) return 0;
    if (host_idx[i] < 0 || host_idx[i] >= host_tokens) return 0;
  }
  return 1;
}

int oracle_backup_all_layers(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                             int64_t device_slots, int64_t host_pages,
                             const uint8_t* const* device_layers, uint8_t* host,
                             const int64_t* device_idx, const int64_t* host_idx, int64_t n) {
  if (!shape_ok(num_layers, page_size, row_bytes, device_slots, host_pages, n)) return ORACLE_BAD_ARG;
  if (n > 0 && (!device_layers || !host || !device_idx || !host_idx)) return ORACLE_BAD_ARG;
  if (!pairs_in_range(device_idx, host_idx, n, device_slots, host_pages * page_size))
    return ORACLE_OUT_OF_RANGE;
  /* The CPU simulation of the staged lf->pf copy: for each layer, the host rows
   * of the destination indices take the device rows of the source indices. */
  for (int64_t l = 0; l < num_layers; ++l) {
    const uint8_t* src_layer = device_layers[l];
    for (int64_t i = 0; i < n; ++i) {
      const uint8_t* src = src_layer + device_row_offset(device_idx[i], row_bytes);
      uint8_t* dst = host + host_row_offset(host_idx[i], l, num_layers, page_size, row_bytes);
      memcpy(dst, src, (size_t)row_bytes);
    }
  }
  return ORACLE_OK;
}

int oracle_load_layer(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                      int64_t device_slots, int64_t host_pages, int64_t layer,
                      uint8_t* device_layer, const uint8_t* host,
                      const int64_t* host_idx, const int64_t* device_idx, int64_t n) {
  if (!shape_ok(num_layers, page_size, row_bytes, device_slots, host_pages, n)) return ORACLE_BAD_ARG;
  if (layer < 0 || layer >= num_layers) return ORACLE_BAD_ARG;
  if (n > 0 && (!device_layer || !host || !device_idx || !host_idx)) return ORACLE_BAD_ARG;
  if (!pairs_in_range(device_idx, host_idx, n, device_slots, host_pages * page_size))
    return ORACLE_OUT_OF_RANGE;
  for (int64_t i = 0; i < n; ++i) {
    const uint8_t* src = host + host_row_offset(host_idx[i], layer, num_layers, page_size, row_bytes);
    uint8_t* dst = device_layer + device_row_offset(device_idx[i], row_bytes);
    memcpy(dst, src, (size_t)row_bytes);
  }
  return ORACLE_OK;
}

int oracle_load_burst(int64_t num_layers, int64_t page_size, int64_t row_bytes,
                      int64_t device_slots, int64_t host_pages,
                      int64_t layer_begin, int64_t layer_end,
                      uint8_t* const* device_layers, const uint8_t* host,
                      const int64_t* host_idx, const int64_t* device_idx, int64_t n) {
  if (layer_begin < 0 || layer_end > num_layers || layer_begin > layer_end) return ORACLE_BAD_ARG;
  if (layer_end > layer_begin && !device_layers) return ORACLE_BAD_ARG;
  for (int64_t l = layer_begin; l < layer_end; ++l) {
    int rc = oracle_load_layer(num_layers, page_size, row_bytes, device_slots, host_pages, l,
                               device_layers[l], host, host_idx, device_idx, n);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

/* ---- page_first host layout: [host token][layer][row] ---------------------- */

/* Byte offset of host token h, layer l, in the token-major host tensor: the
 * staging shape (token, layer, element) of the staged write-back. */
static int64_t pf_host_row_offset(int64_t h, int64_t l, int64_t num_layers, int64_t row_bytes) {
  return (h * num_layers + l) * row_bytes;
}

int oracle_pf_backup_all_layers(int64_t num_layers, int64_t row_bytes, int64_t device_slots,
                                int64_t host_tokens, const uint8_t* const* device_layers,
                                uint8_t* host, const int64_t* device_idx, const int64_t* host_idx,
                                int64_t n) {
  if (!shape_ok(num_layers, 1, row_bytes, device_slots, host_tokens, n)) return ORACLE_BAD_ARG;
  if (n > 0 && (!device_layers || !host || !device_idx || !host_idx)) return ORACLE_BAD_ARG;
  if (!pairs_in_range(device_idx, host_idx, n, device_slots, host_tokens)) return ORACLE_OUT_OF_RANGE;
  /* dst[dst_indices, layer] = src[src_indices], one layer after the other */
  for (int64_t l = 0; l < num_layers; ++l) {
    const uint8_t* src_layer = device_layers[l];
    for (int64_t i = 0; i < n; ++i) {
      const uint8_t* src = src_layer + device_row_offset(device_idx[i], row_bytes);
      uint8_t* dst = host + pf_host_row_offset(host_idx[i], l, num_layers, row_bytes);
      memcpy(dst, src, (size_t)row_bytes);
    }
  }
  return ORACLE_OK;
}

int oracle_pf_load_layer(int64_t num_layers, int64_t row_bytes, int64_t device_slots,
                         int64_t host_tokens, int64_t layer, uint8_t* device_layer,
                         const uint8_t* host, const int64_t* host_idx, const int64_t* device_idx,
                         int64_t n) {
  if (!shape_ok(num_layers, 1, row_bytes, device_slots, host_tokens, n)) return ORACLE_BAD_ARG;
  if (layer < 0 || layer >= num_layers) return ORACLE_BAD_ARG;
  if (n > 0 && (!device_layer || !host || !device_idx || !host_idx)) return ORACLE_BAD_ARG;
  if (!pairs_in_range(device_idx, host_idx, n, device_slots, host_tokens)) return ORACLE_OUT_OF_RANGE;
  for (int64_t i = 0; i < n; ++i) {
    const uint8_t* src = host + pf_host_row_offset(host_idx[i], layer, num_layers, row_bytes);
    uint8_t* dst = device_layer + device_row_offset(device_idx[i], row_bytes);
    memcpy(dst, src, (size_t)row_bytes);
  }
  return ORACLE_OK;
}
