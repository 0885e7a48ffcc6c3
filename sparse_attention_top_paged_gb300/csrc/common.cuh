// common.cuh — device helpers shared by the libidx kernels (sm_103a).
//
// Top-k machinery. Every candidate is a 64-bit composite key
//     key = (order(score) << 32) | (0xFFFFFFFF - index)
// where order() maps float bits to an unsigned integer with the same order
// (-0.0 is folded into +0.0 first). A larger key is a better candidate: higher
// score, then lower index — the output order of the top-k write-out in
// "indexer_score_topk.cu" (score descending, lower index first on ties). Keys
// are unique, so "the k largest keys" is one well-defined set and no tie
// needs a rule beyond the key itself. Key 0 never encodes a real candidate
// and serves as padding.
//
// A TopkGroup is an exact radix select run by a group of NT threads (whole
// warps) of one CTA over keys held in a shared-memory buffer: compact(k)
// keeps exactly the k largest keys, in place, by 8-bit digit histograms.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace idx {

__device__ __forceinline__ uint32_t float_order(float f) {
  uint32_t b = __float_as_uint(__fadd_rn(f, 0.0f));  // -0 + 0 = +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float order_float(uint32_t u) {
  uint32_t b = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(b);
}

__device__ __forceinline__ uint64_t pack_key(float score, int32_t index) {
  return (static_cast<uint64_t>(float_order(score)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(index));
}

__device__ __forceinline__ float key_score(uint64_t key) {
  return order_float(static_cast<uint32_t>(key >> 32));
}

__device__ __forceinline__ int32_t key_index(uint64_t key) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Named barrier over the NT threads of a group (ids 1..15; 0 is __syncthreads).
template <int NT>
__device__ __forceinline__ void group_sync(int bar_id) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(NT) : "memory");
}

struct TopkShared {
  uint32_t hist[256];
  int count;   // entries in the buffer
  int wcount;  // write cursor during compaction
  int sel_bin, sel_above, sel_cnt;
};

template <int NT>
struct TopkGroup {
  TopkShared *s;
  uint64_t *buf;
  int gtid;    // thread index within the group
  int bar_id;  // named barrier of the group

  __device__ __forceinline__ void sync() const { group_sync<NT>(bar_id); }

  // Keep exactly the k largest keys (if more than k are held).
  __device__ void compact(int k) {
    const int n = s->count;
    if (n <= k) return;
    uint64_t prefix = 0, mask = 0;
    int need = k;
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      for (int i = gtid; i < 256; i += NT) s->hist[i] = 0u;
      sync();
      // Four keys per thread per step, loaded before any is used, so a group
      // of a few warps still keeps several shared-memory loads in flight.
      constexpr int U = 4;
      for (int i0 = gtid - static_cast<int>(lane_id()); i0 < n; i0 += U * NT) {
        uint64_t key[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * NT + static_cast<int>(lane_id());
          key[u] = (i < n) ? buf[i] : 0ull;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * NT + static_cast<int>(lane_id());
          const bool part = (i < n) && ((key[u] & mask) == prefix);
          const uint32_t act = __ballot_sync(0xFFFFFFFFu, part);
          if (part) {
            const uint32_t dig = static_cast<uint32_t>(key[u] >> shift) & 255u;
            const uint32_t peers = __match_any_sync(act, dig);
            if (static_cast<int>(lane_id()) == __ffs(peers) - 1) atomicAdd(&s->hist[dig], __popc(peers));
          }
        }
      }
      sync();
      if (gtid < 32) {
        // lane l owns bins 255-8l .. 248-8l, scanned from the top down
        uint32_t c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s->hist[255 - 8 * gtid - j];
          tot += c[j];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (gtid >= o) incl += v;
        }
        uint32_t run = incl - tot;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < static_cast<uint32_t>(need) && run + c[j] >= static_cast<uint32_t>(need)) {
            s->sel_bin = 255 - 8 * gtid - j;
            s->sel_above = static_cast<int>(run);
            s->sel_cnt = static_cast<int>(c[j]);
          }
          run += c[j];
        }
      }
      sync();
      const int bin = s->sel_bin;
      need -= s->sel_above;
      const int cnt = s->sel_cnt;
      prefix |= static_cast<uint64_t>(bin) << shift;
      mask |= 255ull << shift;
      if (cnt == need) break;
    }
    // Keys whose masked prefix is >= prefix are exactly the k largest.
    if (gtid == 0) s->wcount = 0;
    sync();
    constexpr int R = 8;
    for (int base = 0; base < n; base += NT * R) {
      uint64_t v[R];
      bool keep[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int i = base + j * NT + gtid;
        v[j] = (i < n) ? buf[i] : 0ull;
        keep[j] = (i < n) && ((v[j] & mask) >= prefix);
      }
      sync();  // every key of this round is in registers before any write
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep[j]);
        int b = 0;
        if (lane_id() == 0 && m) b = atomicAdd(&s->wcount, __popc(m));
        b = __shfl_sync(0xFFFFFFFFu, b, 0);
        if (keep[j]) buf[b + __popc(m & lanemask_lt())] = v[j];
      }
      // Writes of this round land below base + NT*R (at most as many keys are
      // kept as were read), so the next round's keys are untouched.
    }
    sync();
    if (gtid == 0) s->count = s->wcount;
    sync();
  }
};

}  // namespace idx
