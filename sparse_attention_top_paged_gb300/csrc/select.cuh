// select.cuh — block-wide top-k selection over keys read from memory.
//
// Finds the k largest composite keys (see common.cuh: larger key = higher
// score, then lower index; keys are unique, 0 = no key) among n keys that a
// source yields by index, without buffering them all: a 4096-bin histogram of
// the next 12 key bits locates the bin holding the k-th key; every key above
// that bin is collected directly, and only the keys inside it go through an
// exact radix select in shared memory. If that bin is still larger than the
// boundary buffer (many keys sharing the same leading bits, e.g. equal
// scores), the bin is refined with the next 12 bits, re-reading the source.
//
// Src must provide `void begin()` (called before each pass over the source)
// and `uint64_t get(int i)` for i in [0, n); passes read i = tid, tid + NT, ...
// in increasing order per thread, kU of them before using any.
#pragma once

#include "common.cuh"

namespace idx {

constexpr int kSelBins = 4096;
constexpr int kU = 8;  // keys each thread loads before using any of them

struct SelectShared {
  uint32_t hist[kSelBins];
  uint32_t warp_sum[32];
  int bin, above, bin_cnt, total;
  int n_out, n_bnd;
};

template <int NT>
struct BlockSelect {
  static_assert(NT % 32 == 0 && NT <= 1024 && kSelBins % NT == 0, "block shape");
  SelectShared *sh;
  TopkShared *tsh;   // exact select of the boundary bin
  uint64_t *out;     // >= k keys
  uint64_t *bnd;     // boundary buffer
  int bnd_cap;       // >= NT
  int bar_id;

  __device__ __forceinline__ void sync() const { group_sync<NT>(bar_id); }

  // Warp-aggregated append of `key` (when `take`) to buf[*cnt ...]. Every lane
  // of the warp must call it.
  __device__ __forceinline__ void append(uint64_t *buf, int *cnt, uint64_t key, bool take) const {
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
    int base = 0;
    if (lane_id() == 0 && m) base = atomicAdd(cnt, __popc(m));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (take) buf[base + __popc(m & lanemask_lt())] = key;
  }

  // Returns the number of keys selected (min(k, valid keys)); out[0 .. count)
  // holds them, unordered.
  template <class Src>
  __device__ int run(Src &src, int n, int k) {
    const int tid = static_cast<int>(threadIdx.x) % NT;
    uint64_t prefix = 0, mask = 0;
    int need = k;
    int shift = 52;
    bool take_all = false;
    int width = 12;
    while (true) {
      for (int b = tid; b < kSelBins; b += NT) sh->hist[b] = 0u;
      if (tid == 0) sh->total = 0;
      sync();
      src.begin();
      const uint32_t dmask = (1u << width) - 1u;
      for (int i0 = tid - static_cast<int>(lane_id()); i0 < n; i0 += kU * NT) {
        uint64_t key[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {   // all loads first: one memory latency per kU keys
          const int i = i0 + u * NT + static_cast<int>(lane_id());
          key[u] = (i < n) ? src.get(i) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (key[u] != 0ull && (key[u] & mask) == prefix)
            atomicAdd(&sh->hist[static_cast<uint32_t>(key[u] >> shift) & dmask], 1u);
        }
      }
      sync();
      // Bins in descending order: thread tid owns bins kSelBins-1-per*tid-j, j < per.
      constexpr int per = kSelBins / NT;
      uint32_t c[per], tot = 0;
#pragma unroll
      for (int j = 0; j < per; ++j) {
        c[j] = sh->hist[kSelBins - 1 - per * tid - j];
        tot += c[j];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane_id() >= static_cast<uint32_t>(o)) incl += v;
      }
      if (lane_id() == 31) sh->warp_sum[tid >> 5] = incl;
      sync();
      uint32_t before = 0, all = 0;
      for (int wi = 0; wi < NT / 32; ++wi) {
        const uint32_t s = sh->warp_sum[wi];
        if (wi < (tid >> 5)) before += s;
        all += s;
      }
      uint32_t run = before + incl - tot;
      if (all <= static_cast<uint32_t>(need)) {
        take_all = true;            // every key matching the prefix is selected
      } else {
#pragma unroll
        for (int j = 0; j < per; ++j) {
          if (run < static_cast<uint32_t>(need) && run + c[j] >= static_cast<uint32_t>(need)) {
            sh->bin = kSelBins - 1 - per * tid - j;
            sh->above = static_cast<int>(run);
            sh->bin_cnt = static_cast<int>(c[j]);
          }
          run += c[j];
        }
      }
      sync();
      if (take_all) break;
      const int bin = sh->bin;
      if (sh->bin_cnt <= bnd_cap || shift == 0) {
        prefix |= static_cast<uint64_t>(bin) << shift;
        mask |= static_cast<uint64_t>(dmask) << shift;
        break;
      }
      // refine the boundary bin with the next digit
      need -= sh->above;
      prefix |= static_cast<uint64_t>(bin) << shift;
      mask |= static_cast<uint64_t>(dmask) << shift;
      // digits: bits 63..52, 51..40, 39..28, 27..16, 15..4, then 3..0
      if (shift >= 12) {
        shift -= 12;
        width = 12;
      } else {
        width = shift;
        shift = 0;
      }
      sync();
    }
    // Collect: keys above the boundary go to out; keys in it to bnd.
    if (tid == 0) {
      sh->n_out = 0;
      sh->n_bnd = 0;
    }
    sync();
    src.begin();
    for (int i0 = tid - static_cast<int>(lane_id()); i0 < n; i0 += kU * NT) {
      uint64_t key[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * NT + static_cast<int>(lane_id());
        key[u] = (i < n) ? src.get(i) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint64_t mk = key[u] & mask;
        const bool up = key[u] != 0ull && (take_all ? mk >= prefix : mk > prefix);
        const bool eq = key[u] != 0ull && !take_all && mk == prefix;
        append(out, &sh->n_out, key[u], up);
        append(bnd, &sh->n_bnd, key[u], eq);
      }
    }
    sync();
    int count = sh->n_out;
    if (!take_all) {
      const int nb = sh->n_bnd;
      const int want = k - count;   // 1 .. nb
      TopkGroup<NT> g{tsh, bnd, bnd_cap, tid, bar_id};
      if (tid == 0) tsh->count = nb;
      sync();
      g.compact(want);               // keeps the `want` largest boundary keys in bnd[0 .. want)
      for (int i = tid; i < want; i += NT) out[count + i] = bnd[i];
      sync();
      count += want;
    }
    return count;
  }

  // Sort out[0 .. count) descending (count <= cap2, a power of two >= count
  // fits in out), padding with key 0.
  __device__ void sort_desc(int count) {
    const int tid = static_cast<int>(threadIdx.x) % NT;
    int m = 1;
    while (m < count) m <<= 1;
    for (int i = count + tid; i < m; i += NT) out[i] = 0ull;
    sync();
    for (int size = 2; size <= m; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < (m >> 1); i += NT) {
          const int lo = 2 * stride * (i / stride) + (i % stride);
          const int hi = lo + stride;
          const bool desc = (lo & size) == 0;
          const uint64_t a = out[lo], b = out[hi];
          if ((a < b) == desc) {
            out[lo] = b;
            out[hi] = a;
          }
        }
        sync();
      }
    }
  }
};

}  // namespace idx
