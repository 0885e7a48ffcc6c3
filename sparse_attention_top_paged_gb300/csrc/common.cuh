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

#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/idx.h"

namespace idx {

// Index checks of debug-bounds builds (-DIDX_DEBUG_BOUNDS): a failed check ORs
// IDX_STATUS_DEBUG_BOUNDS into the status word and the access it guards is
// skipped. In other builds a check is the constant true and compiles away.
#ifdef IDX_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, int32_t *status) {
  if (!ok && status != nullptr) atomicOr(status, IDX_STATUS_DEBUG_BOUNDS);
  return ok;
}
#define IDX_IN_BOUNDS(cond, status) ::idx::in_bounds((cond), (status))
#else
#define IDX_IN_BOUNDS(cond, status) true
#endif

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

}  // namespace idx
