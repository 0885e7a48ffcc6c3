// static_scratch.cu — idx_score_topk_static: idx_score_topk without a
// caller-provided workspace.
//
// Some callers cannot call cudaMalloc at all: a plugin running inside a host
// runtime that owns every byte of device memory and hands its operators no
// allocator, or a serving loop that must not allocate after start-up (an
// allocation can block on the device and can fail under memory pressure at
// an unpredictable moment). For them this entry point runs the same kernels
// as idx_score_topk on a scratch array that lives in the library itself: a
// file-scope __device__ array of IDX_STATIC_SCRATCH_BYTES bytes, which every
// GPU that loads libidx holds until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// only names a stand-in object), so the first call on each device, with that
// device current, asks the runtime for the array's device address with
// cudaGetSymbolAddress and caches it; later calls reuse it. That first call
// should therefore come before any stream capture.
//
// Every call shares the one array and leaves its last contents behind.
// Nothing in it has to start at zero: each call writes every scratch word it
// reads. Calls whose execution overlaps on the GPU (different streams, or
// different host threads without ordering) race on the array.
#include <mutex>
#include <vector>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[IDX_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device (set up once per
// device). Returns nullptr if the runtime cannot provide it.
void *static_scratch_address() {
  static std::mutex mu;
  static std::vector<void *> addr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(addr.size()) <= dev) addr.resize(dev + 1, nullptr);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" idx_status_t idx_score_topk_static(const idx_score_topk_args *args, idx_stream_t stream) {
  if (!args) return IDX_ERR_INVALID_ARG;
  idx_score_topk_args a = *args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  size_t need = 0;
  const idx_status_t st = idx_score_topk_workspace_size(&a, &need);
  if (st != IDX_OK) return st;
  if (need > IDX_STATIC_SCRATCH_BYTES) return IDX_ERR_WORKSPACE_TOO_SMALL;
  if (a.T == 0) return IDX_OK;
  void *scratch = static_scratch_address();
  if (scratch == nullptr) return IDX_ERR_CUDA;
  a.workspace = scratch;
  a.workspace_bytes = IDX_STATIC_SCRATCH_BYTES;
  return idx_score_topk(&a, stream);
}
