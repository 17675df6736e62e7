// validate.cpp -- host-side argument checks and the run planner.
//
// Everything here is plain C++ and calls no CUDA function, so it runs (and is
// tested) on machines without a GPU.  Index validation replaces the per-chunk
// copy-descriptor build that the per-layer load performs on the CPU in the
// HiCache pages ("[HiCache] Run the host->device load-back enqueue on a loader
// thread", Motivation): one O(n) pass per call or per burst, then nothing per
// layer.
#include <algorithm>
#include <cstring>
#include <limits>
#include <string>
#include <vector>

#include "hicache_internal.h"

namespace hk {

namespace {
thread_local std::string g_last_error;

template <typename T>
inline int64_t idx_at(const void* p, int64_t i) {
  return static_cast<int64_t>(static_cast<const T*>(p)[i]);
}

inline int64_t idx(const void* p, int32_t bits, int64_t i) {
  return bits == 32 ? idx_at<int32_t>(p, i) : idx_at<int64_t>(p, i);
}

std::string str(int64_t v) { return std::to_string(v); }

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

template <typename T>
void min_max(const T* p, int64_t n, int64_t* mn, int64_t* mx) {
  T lo = p[0], hi = p[0];
  for (int64_t i = 1; i < n; ++i) {
    lo = p[i] < lo ? p[i] : lo;
    hi = p[i] > hi ? p[i] : hi;
  }
  *mn = int64_t(lo);
  *mx = int64_t(hi);
}

// End of the run that starts at pair i: the first j > i at which d or h does
// not step by one from pair j - 1 (or n).  Differences are taken modulo 2^64,
// which is defined for every value; a run that wraps past the largest int64 is
// caught by the range check (its last value is below its first).  Blocks of 8
// pairs are tested without branches, so a long run costs a fraction of a
// nanosecond per pair, and a run of one pair a single comparison.
template <typename T>
int64_t run_end(const T* d, const T* h, int64_t i, int64_t n) {
  auto steps = [&](int64_t j) {
    return (uint64_t(int64_t(d[j])) - uint64_t(int64_t(d[j - 1])) - 1u) |
           (uint64_t(int64_t(h[j])) - uint64_t(int64_t(h[j - 1])) - 1u);
  };
  int64_t j = i + 1;
  if (j < n && steps(j) != 0) return j;
  while (j + 8 <= n) {
    uint64_t off = 0;
    for (int u = 0; u < 8; ++u) off |= steps(j + u);
    if (off != 0) break;
    j += 8;
  }
  while (j < n && steps(j) == 0) ++j;
  return j;
}

// Marks rows [x0, x0 + len) in the bitmap a word at a time.  Returns the first
// row of the range that was already marked (nothing past it is marked then), or
// -1.
int64_t mark_range(uint64_t* bitmap, int64_t x0, int64_t len) {
  const int64_t end = x0 + len;
  for (int64_t x = x0; x < end;) {
    const int b = int(x & 63);
    const int64_t take = std::min<int64_t>(64 - b, end - x);
    const uint64_t mask = (take == 64 ? ~uint64_t(0) : (uint64_t(1) << take) - 1) << b;
    uint64_t& w = bitmap[x >> 6];
    if (w & mask) return (x & ~int64_t(63)) + __builtin_ctzll(w & mask);
    w |= mask;
    x += take;
  }
  return -1;
}

// Result of the run pass over a pair list.
struct RunCheck {
  bool out_of_range = false;  // some pair addresses no row (named by a second walk)
  int64_t dup_pair = -1;      // first pair whose destination was already named
  int64_t dup_row = -1;       // that destination
  int64_t bad_page = -1;      // first pair that breaks the whole-page structure
  bool bad_start = false;     // ... because its page does not start page-aligned
};

// One pass over the runs of the pair list (maximal stretches where both sides
// step by one).  Within a run the indices grow by one, so its first and last
// pairs decide its range.  Destinations are marked in the bitmap run by run;
// after the first duplicate only ranges are still checked, since a range error
// takes precedence.  With `pages` every run must start a page in pair order and
// page-aligned on both sides, which is exactly "every group of P pairs is one
// whole aligned page" once n is a multiple of P.  The bitmap is left all zero.
template <typename T>
RunCheck check_runs(const T* d, const T* h, int64_t n, bool dest_is_device, bool pages, int64_t P,
                    int64_t dev_lim, int64_t host_lim, uint64_t* bitmap) {
  const T* dst = dest_is_device ? d : h;
  RunCheck rc;
  int64_t marked_end = 0;  // pairs [0, marked_end) may have marked words
  int64_t lo = std::numeric_limits<int64_t>::max(), hi = -1;  // destinations marked
  for (int64_t i = 0; i < n;) {
    const int64_t e = run_end(d, h, i, n);
    const int64_t d0 = int64_t(d[i]), d1 = int64_t(d[e - 1]);
    const int64_t h0 = int64_t(h[i]), h1 = int64_t(h[e - 1]);
    if (d0 < 0 || d1 >= dev_lim || d1 < d0 || h0 < 0 || h1 >= host_lim || h1 < h0) {
      rc.out_of_range = true;
      break;
    }
    if (pages && rc.bad_page < 0) {
      if (i % P != 0) {
        rc.bad_page = i;
      } else if (d0 % P != 0 || h0 % P != 0) {
        rc.bad_page = i;
        rc.bad_start = true;
      }
    }
    if (rc.dup_pair < 0) {
      const int64_t x0 = dest_is_device ? d0 : h0;
      int64_t hit = -1;
      if (e == i + 1) {  // a run of one pair: one bit
        uint64_t& w = bitmap[x0 >> 6];
        const uint64_t bit = uint64_t(1) << (x0 & 63);
        if (w & bit) hit = x0;
        w |= bit;
      } else {
        hit = mark_range(bitmap, x0, e - i);
      }
      marked_end = e;
      lo = std::min(lo, x0);
      hi = std::max(hi, x0 + (e - i) - 1);
      if (hit >= 0) {
        rc.dup_pair = i + (hit - x0);
        rc.dup_row = hit;
      }
    }
    i = e;
  }
  // Clear what was marked: every word of [lo, hi] when that is no more words
  // than pairs, else the word of each pair marked.
  if (hi >= lo && (hi >> 6) - (lo >> 6) + 1 <= n) {
    std::fill(bitmap + (lo >> 6), bitmap + (hi >> 6) + 1, uint64_t(0));
  } else {
    for (int64_t j = 0; j < marked_end; ++j) bitmap[int64_t(dst[j]) >> 6] = 0;
  }
  return rc;
}
}  // namespace

hicache_status check_whole_pages(bool any_page, int64_t P, const void* dev_idx, const void* host_idx,
                                 int32_t bits, int64_t n);

void set_error(const std::string& msg) { g_last_error = msg; }
void clear_error() { g_last_error.clear(); }
hicache_status fail(hicache_status st, const std::string& msg) {
  set_error(msg);
  return st;
}
const std::string& last_error() { return g_last_error; }

hicache_status check_pools(const hicache_pool* pools, int32_t num_pools, std::vector<PoolInfo>* out) {
  if (!pools) return fail(HICACHE_EINVAL, "pools is NULL");
  if (num_pools < 1 || num_pools > kMaxPools)
    return fail(HICACHE_EINVAL, "num_pools must be in 1.." + str(kMaxPools));
  out->clear();
  for (int32_t p = 0; p < num_pools; ++p) {
    const hicache_pool& q = pools[p];
    const std::string who = "pool " + str(p) + ": ";
    if (q.num_layers < 1 || q.num_layers > 4096) return fail(HICACHE_EINVAL, who + "num_layers must be in 1..4096");
    if (q.num_tensors < 1 || q.num_tensors > 2) return fail(HICACHE_EINVAL, who + "num_tensors must be 1 or 2");
    if (q.head_num < 1 || q.head_dim < 1 || q.dtype_size < 1)
      return fail(HICACHE_EINVAL, who + "head_num, head_dim and dtype_size must be positive");
    if (q.page_size < 1) return fail(HICACHE_EINVAL, who + "page_size must be positive");
    if (q.page_granular != 0 && q.page_granular != 1) return fail(HICACHE_EINVAL, who + "page_granular must be 0 or 1");
    if (q.layout != HICACHE_LAYOUT_PAGE_FIRST_DIRECT && q.layout != HICACHE_LAYOUT_PAGE_FIRST)
      return fail(HICACHE_EINVAL, who + "layout is not a hicache_layout");
    const int64_t R = int64_t(q.head_num) * q.head_dim * q.dtype_size;
    if (R > (int64_t(1) << 24)) return fail(HICACHE_EINVAL, who + "row bytes above 16 MiB");
    if (R % 4 != 0) return fail(HICACHE_EALIGN, who + "row bytes " + str(R) + " not a multiple of 4");
    if (q.device_slots < 0 || q.host_pages < 0) return fail(HICACHE_EINVAL, who + "negative pool size");
    if (q.device_slots > kMaxRows || q.host_pages * int64_t(q.page_size) > kMaxRows)
      return fail(HICACHE_EINVAL, who + "pool holds more than 2^31-1 token rows");
    if (q.page_granular && q.device_slots % q.page_size != 0)
      return fail(HICACHE_EINVAL, who + "page-granular pool: device_slots not a multiple of page_size");
    if (q.page_granular && int64_t(q.page_size) * R > (int64_t(1) << 24))
      return fail(HICACHE_EINVAL, who + "page row above 16 MiB");
    if (!q.device_layers || !q.host_tensors) return fail(HICACHE_EINVAL, who + "NULL pointer table");
    PoolInfo pi;
    pi.L = q.num_layers;
    pi.T = q.num_tensors;
    pi.P = q.page_size;
    pi.page_granular = q.page_granular;
    pi.layout = q.layout;
    pi.token_bytes = R;
    pi.device_slots = q.device_slots;
    pi.host_pages = q.host_pages;
    pi.dev.resize(size_t(pi.T) * pi.L);
    pi.host.resize(size_t(pi.T));
    for (int32_t i = 0; i < pi.T * pi.L; ++i) {
      char* ptr = static_cast<char*>(q.device_layers[i]);
      if (!ptr) return fail(HICACHE_EINVAL, who + "device layer pointer " + str(i) + " is NULL");
      if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0)
        return fail(HICACHE_EALIGN, who + "device layer pointer " + str(i) + " not 4-byte aligned");
      pi.dev[size_t(i)] = ptr;
    }
    for (int32_t t = 0; t < pi.T; ++t) {
      char* ptr = static_cast<char*>(q.host_tensors[t]);
      if (!ptr) return fail(HICACHE_EINVAL, who + "host tensor pointer " + str(t) + " is NULL");
      if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0)
        return fail(HICACHE_EALIGN, who + "host tensor pointer " + str(t) + " not 4-byte aligned");
      pi.host[size_t(t)] = ptr;
    }
    out->push_back(std::move(pi));
  }
  for (size_t p = 1; p < out->size(); ++p) {
    if ((*out)[p].L != (*out)[0].L)
      return fail(HICACHE_EINVAL, "pools of one call must have the same num_layers");
    if ((*out)[p].P != (*out)[0].P)
      return fail(HICACHE_EINVAL, "pools of one call must have the same page_size");
  }
  return HICACHE_OK;
}

hicache_status check_index_args(const void* a, const void* b, int32_t index_bits, int64_t n) {
  if (index_bits != 32 && index_bits != 64) return fail(HICACHE_EINVAL, "index_bits must be 32 or 64");
  if (n < 0) return fail(HICACHE_EINVAL, "n is negative");
  if (n > kMaxRows) return fail(HICACHE_EINVAL, "n above 2^31-1");
  if (n > 0 && (!a || !b)) return fail(HICACHE_EINVAL, "NULL index array");
  return HICACHE_OK;
}

hicache_status check_pairs_host(const std::vector<PoolInfo>& pools, const void* dev_idx,
                                const void* host_idx, int32_t bits, int64_t n, bool dest_is_device) {
  if (n == 0) return HICACHE_OK;
  int64_t dev_lim = std::numeric_limits<int64_t>::max();
  int64_t host_lim = std::numeric_limits<int64_t>::max();
  bool any_page = false;
  const int64_t P = pools[0].P;
  for (const PoolInfo& p : pools) {
    dev_lim = std::min(dev_lim, p.device_slots);
    host_lim = std::min(host_lim, p.host_pages * int64_t(p.P));
    any_page = any_page || p.page_granular;
  }
  const void* dst = dest_is_device ? dev_idx : host_idx;
  const int64_t lim = dest_is_device ? dev_lim : host_lim;
  // Names the first pair that addresses no row of every pool of the call.
  auto range_error = [&]() {
    for (int64_t i = 0; i < n; ++i) {
      const int64_t d = idx(dev_idx, bits, i);
      const int64_t h = idx(host_idx, bits, i);
      if (d < 0 || d >= dev_lim)
        return fail(HICACHE_ERANGE, "device index " + str(d) + " at pair " + str(i) + " outside [0, " + str(dev_lim) + ")");
      if (h < 0 || h >= host_lim)
        return fail(HICACHE_ERANGE, "host index " + str(h) + " at pair " + str(i) + " outside [0, " + str(host_lim) + ")");
    }
    return fail(HICACHE_ERANGE, "index out of range");  // not reached
  };
  if (lim > (int64_t(1) << 28) && lim / 64 > 4 * n) {
    // Sparse use of a huge destination space: a min/max pass for the range,
    // then distinct destinations by sorting a copy instead of a bitmap.
    int64_t dmin, dmax, hmin, hmax;
    if (bits == 32) {
      min_max(static_cast<const int32_t*>(dev_idx), n, &dmin, &dmax);
      min_max(static_cast<const int32_t*>(host_idx), n, &hmin, &hmax);
    } else {
      min_max(static_cast<const int64_t*>(dev_idx), n, &dmin, &dmax);
      min_max(static_cast<const int64_t*>(host_idx), n, &hmin, &hmax);
    }
    if (dmin < 0 || dmax >= dev_lim || hmin < 0 || hmax >= host_lim) return range_error();
    std::vector<int64_t> v(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) v[size_t(i)] = idx(dst, bits, i);
    std::sort(v.begin(), v.end());
    for (size_t i = 1; i < v.size(); ++i)
      if (v[i] == v[i - 1])
        return fail(HICACHE_EDUP, std::string(dest_is_device ? "device" : "host") + " destination " +
                                      str(v[i]) + " named twice");
    return check_whole_pages(any_page, P, dev_idx, host_idx, bits, n);
  }
  // Range, distinct destinations (a bitmap over the destination rows, cleared
  // again after use so that the cost stays O(n) per call) and whole pages, in
  // one pass over the runs of the pair list.
  static thread_local std::vector<uint64_t> bitmap;
  const size_t words = size_t((lim + 63) / 64);
  if (bitmap.size() < words) bitmap.assign(words, 0);
  const RunCheck rc = bits == 32
      ? check_runs(static_cast<const int32_t*>(dev_idx), static_cast<const int32_t*>(host_idx), n,
                   dest_is_device, any_page, P, dev_lim, host_lim, bitmap.data())
      : check_runs(static_cast<const int64_t*>(dev_idx), static_cast<const int64_t*>(host_idx), n,
                   dest_is_device, any_page, P, dev_lim, host_lim, bitmap.data());
  if (rc.out_of_range) return range_error();
  if (rc.dup_pair >= 0)
    return fail(HICACHE_EDUP, std::string(dest_is_device ? "device" : "host") + " destination " +
                                  str(rc.dup_row) + " named twice (second time at pair " +
                                  str(rc.dup_pair) + ")");
  if (any_page && n % P != 0)
    return fail(HICACHE_EINVAL, "page-granular pool: n=" + str(n) + " is not a multiple of page_size " + str(P));
  if (rc.bad_page >= 0) {
    const int64_t k = rc.bad_page / P * P;
    if (rc.bad_start)
      return fail(HICACHE_EINVAL, "page-granular pool: pair " + str(k) + " does not start a page");
    return fail(HICACHE_EINVAL, "page-granular pool: pairs " + str(k) + ".." + str(k + P - 1) +
                                    " are not one whole page");
  }
  return HICACHE_OK;
}

hicache_status check_whole_pages(bool any_page, int64_t P, const void* dev_idx, const void* host_idx,
                                 int32_t bits, int64_t n) {
  // Page-granular pools move whole aligned pages.
  if (any_page) {
    if (n % P != 0)
      return fail(HICACHE_EINVAL, "page-granular pool: n=" + str(n) + " is not a multiple of page_size " + str(P));
    for (int64_t k = 0; k < n; k += P) {
      const int64_t d0 = idx(dev_idx, bits, k);
      const int64_t h0 = idx(host_idx, bits, k);
      if (d0 % P != 0 || h0 % P != 0)
        return fail(HICACHE_EINVAL, "page-granular pool: pair " + str(k) + " does not start a page");
      for (int64_t t = 1; t < P; ++t) {
        if (idx(dev_idx, bits, k + t) != d0 + t || idx(host_idx, bits, k + t) != h0 + t)
          return fail(HICACHE_EINVAL, "page-granular pool: pairs " + str(k) + ".." + str(k + P - 1) +
                                          " are not one whole page");
      }
    }
  }
  return HICACHE_OK;
}

hicache_status plan_runs(const void* dev_idx, const void* host_idx, int32_t bits, int64_t n,
                         int32_t page_size, hicache_run* runs, int64_t cap, int64_t* num_runs,
                         int64_t* full_pages) {
  if (page_size < 1) return fail(HICACHE_EINVAL, "page_size must be positive");
  if (!num_runs) return fail(HICACHE_EINVAL, "num_runs is NULL");
  if (cap < 0) return fail(HICACHE_EINVAL, "runs_cap is negative");
  const int64_t P = page_size;
  int64_t count = 0, full = 0;
  // Maximal stretches where both sides step by one, cut where the host slot
  // starts a new page.
  auto plan = [&](const auto* d, const auto* h) {
    for (int64_t i = 0; i < n;) {
      const int64_t e = run_end(d, h, i, n);
      for (int64_t s = i; s < e;) {
        const int64_t h0 = int64_t(h[s]);
        const int64_t to_page_end = P - ((h0 % P) + P) % P;  // pairs left in h0's page
        const int64_t len = std::min(e - s, to_page_end);
        if (runs && count < cap) runs[count] = hicache_run{int64_t(d[s]), h0, len};
        if (len == P && h0 % P == 0) ++full;
        ++count;
        s += len;
      }
      i = e;
    }
  };
  if (bits == 32) plan(static_cast<const int32_t*>(dev_idx), static_cast<const int32_t*>(host_idx));
  else plan(static_cast<const int64_t*>(dev_idx), static_cast<const int64_t*>(host_idx));
  *num_runs = count;
  if (full_pages) *full_pages = full;
  return HICACHE_OK;
}

}  // namespace hk
