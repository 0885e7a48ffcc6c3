// gather_split.cu — the dense-tile gather of "Commit graph,
// dsv4/kernels/indexer" (commit c2f705a, gather_kv.cu): selected positions of
// a paged cache whose rows are split into an FP8 part ("nope") and a BF16 part
// ("rope"), resolved through the block table, the FP8 part dequantised to BF16,
// written as one dense BF16 tile for the attention that follows.
//
// The commit gives no layout; the one taken here: per token nope_dim E4M3
// bytes ([P, block_size, nope_dim]), an optional FP32 scale per token
// ([P, block_size]), rope_dim BF16 values ([P, block_size, rope_dim]);
// out[t, i] = [bf16_rn(float(e4m3) * scale) for the nope part, the rope part
// unchanged]. Positions resolve exactly as idx_gather_kv resolves them. One
// warp per output row.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kSplitWarps = 8;

__device__ __forceinline__ uint32_t dequant2(uint32_t two_bytes, float scale) {
  const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes), __NV_E4M3);
  const float lo = __half2float(__half(__half_raw{h2.x})) * scale;
  const float hi = __half2float(__half(__half_raw{h2.y})) * scale;
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // each half rounded to nearest even
  return *reinterpret_cast<const uint32_t *>(&b);
}

__global__ void __launch_bounds__(kSplitWarps * 32) gather_split_kernel(idx_gather_split_args a) {
  const long long r = static_cast<long long>(blockIdx.x) * kSplitWarps + (threadIdx.x >> 5);
  const long long n_rows = static_cast<long long>(a.T) * a.n_sel;
  if (r >= n_rows) return;
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>(r / a.n_sel);
  const int pos = a.sel[r];
  long long src = -1;
  int err = 0;
  if (pos >= 0) {
    const int lb = pos / a.block_size;
    if (lb >= a.max_logical_blocks) {
      err = IDX_STATUS_BAD_SEL;
    } else {
      const int phys = a.block_table[static_cast<long long>(t) * a.bt_stride + lb];
      if (phys < 0 || phys >= a.P)
        err = IDX_STATUS_BAD_BLOCK;
      else
        src = static_cast<long long>(phys) * a.block_size + pos % a.block_size;
    }
  }
  if (err && lane == 0 && a.dev_status) atomicOr(a.dev_status, err);
  if (src >= 0 && !IDX_IN_BOUNDS(src < static_cast<long long>(a.P) * a.block_size, a.dev_status)) src = -1;
  const int width = a.nope_dim + a.rope_dim;   // even
  uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + r * width);
  if (src < 0) {
    for (int i = lane; i < width / 2; i += 32) dst[i] = 0u;
    return;
  }
  const float scale = a.nope_scale ? a.nope_scale[src] : 1.0f;
  const uint32_t *nope = reinterpret_cast<const uint32_t *>(a.nope + src * a.nope_dim);
  for (int i = lane; i < a.nope_dim / 4; i += 32) {   // four E4M3 values -> two bf16 pairs
    const uint32_t w = __ldg(nope + i);
    dst[2 * i] = dequant2(w & 0xFFFFu, scale);
    dst[2 * i + 1] = dequant2(w >> 16, scale);
  }
  const uint32_t *rope = reinterpret_cast<const uint32_t *>(a.rope + src * a.rope_dim);
  for (int i = lane; i < a.rope_dim / 2; i += 32) dst[a.nope_dim / 2 + i] = __ldg(rope + i);
}

// The same rows when the nope part is a whole number of 8-byte pieces, the
// rope part of 8 values, and every pointer 16-byte aligned: a warp takes
// kVecRows rows and looks both up at once; a lane then reads 8 E4M3 bytes of
// two pieces of each row (all loads issued before any is converted) and writes
// each piece's 16 output bytes, so a warp's stores are contiguous and a warp
// has both rows' bytes in flight. The arithmetic is the kernel's above, pair
// by pair.
constexpr int kVecRows = 8;

__device__ __forceinline__ uint4 ldg16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

__global__ void __launch_bounds__(kSplitWarps * 32) gather_split_vec_kernel(idx_gather_split_args a) {
  const long long r0 = (static_cast<long long>(blockIdx.x) * kSplitWarps + (threadIdx.x >> 5)) * kVecRows;
  const long long n_rows = static_cast<long long>(a.T) * a.n_sel;
  if (r0 >= n_rows) return;
  const int lane = threadIdx.x & 31;
  // lane i < kVecRows resolves row r0 + i
  long long my_src = -1;
  if (lane < kVecRows && r0 + lane < n_rows) {
    const long long r = r0 + lane;
    const int t = static_cast<int>(r / a.n_sel);
    const int pos = a.sel[r];
    int err = 0;
    if (pos >= 0) {
      const int lb = pos / a.block_size;
      if (lb >= a.max_logical_blocks) {
        err = IDX_STATUS_BAD_SEL;
      } else {
        const int phys = a.block_table[static_cast<long long>(t) * a.bt_stride + lb];
        if (phys < 0 || phys >= a.P)
          err = IDX_STATUS_BAD_BLOCK;
        else
          my_src = static_cast<long long>(phys) * a.block_size + pos % a.block_size;
      }
    }
    if (err && a.dev_status) atomicOr(a.dev_status, err);
    if (my_src >= 0 && !IDX_IN_BOUNDS(my_src < static_cast<long long>(a.P) * a.block_size, a.dev_status)) my_src = -1;
  }
  long long src[kVecRows];
  float scale[kVecRows];
#pragma unroll
  for (int i = 0; i < kVecRows; ++i) {
    src[i] = (r0 + i < n_rows) ? __shfl_sync(0xFFFFFFFFu, my_src, i) : -2;   // -2: no such row
    scale[i] = (src[i] >= 0 && a.nope_scale) ? a.nope_scale[src[i]] : 1.0f;
  }
  const int width = a.nope_dim + a.rope_dim;
  const int nope8 = a.nope_dim / 8, rope8 = a.rope_dim / 8;   // pieces of 8 values: 8 bytes in (E4M3), 16 out
  constexpr int kU = 2;                                        // pieces a lane takes at once (per row)
  for (int c0 = 0; c0 < nope8; c0 += 32 * kU) {
    uint2 v[kVecRows][kU];
#pragma unroll
    for (int i = 0; i < kVecRows; ++i)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u + lane;
        v[i][u] = (src[i] >= 0 && c < nope8)
                      ? __ldg(reinterpret_cast<const uint2 *>(a.nope + src[i] * a.nope_dim + 8 * c))
                      : make_uint2(0u, 0u);
      }
#pragma unroll
    for (int i = 0; i < kVecRows; ++i)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u + lane;
        if (src[i] == -2 || c >= nope8) continue;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (src[i] >= 0)
          o = make_uint4(dequant2(v[i][u].x & 0xFFFFu, scale[i]), dequant2(v[i][u].x >> 16, scale[i]),
                         dequant2(v[i][u].y & 0xFFFFu, scale[i]), dequant2(v[i][u].y >> 16, scale[i]));
        reinterpret_cast<uint4 *>(a.out + (r0 + i) * width)[c] = o;   // a warp's stores: 512 contiguous bytes
      }
  }
  for (int c0 = 0; c0 < rope8; c0 += 32) {   // 8 bf16 values a piece, copied
    const int c = c0 + lane;
    uint4 v[kVecRows];
#pragma unroll
    for (int i = 0; i < kVecRows; ++i)
      v[i] = (src[i] >= 0 && c < rope8) ? ldg16(a.rope + (src[i] * a.rope_dim + 8 * c)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < kVecRows; ++i)
      if (src[i] != -2 && c < rope8) reinterpret_cast<uint4 *>(a.out + (r0 + i) * width + a.nope_dim)[c] = v[i];
  }
}

bool aligned4(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }
bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace
}  // namespace idx

extern "C" idx_status_t idx_gather_split(const idx_gather_split_args *a, idx_stream_t stream) {
  using namespace idx;
  if (!a) return IDX_ERR_INVALID_ARG;
  if (a->T < 0 || a->n_sel < 0 || a->max_logical_blocks < 1 || a->bt_stride < 0 || a->P < 1 || a->block_size < 1 ||
      a->nope_dim < 0 || a->rope_dim < 0 || a->nope_dim % 4 != 0 || a->rope_dim % 2 != 0 ||
      a->nope_dim + a->rope_dim == 0)
    return IDX_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(a->T) * a->n_sel;
  if (rows == 0) return IDX_OK;
  if (!a->sel || !a->block_table || !a->out || (a->nope_dim > 0 && !a->nope) || (a->rope_dim > 0 && !a->rope))
    return IDX_ERR_INVALID_ARG;
  if (!aligned4(a->sel) || !aligned4(a->block_table) || !aligned4(a->out) || (a->nope && !aligned4(a->nope)) ||
      (a->rope && !aligned4(a->rope)) || (a->nope_scale && !aligned4(a->nope_scale)) ||
      (a->dev_status && !aligned4(a->dev_status)))
    return IDX_ERR_INVALID_ARG;
  if ((rows + kSplitWarps - 1) / kSplitWarps > 0x7FFFFFFFLL) return IDX_ERR_UNSUPPORTED;
  const bool vec = a->nope_dim % 8 == 0 && a->rope_dim % 8 == 0 && aligned16(a->out) &&
                   (a->nope_dim == 0 || aligned16(a->nope)) && (a->rope_dim == 0 || aligned16(a->rope));
  if (vec) {
    const long long per_block = static_cast<long long>(kSplitWarps) * kVecRows;
    const unsigned grid = static_cast<unsigned>((rows + per_block - 1) / per_block);
    gather_split_vec_kernel<<<grid, kSplitWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(*a);
  } else {
    const unsigned grid = static_cast<unsigned>((rows + kSplitWarps - 1) / kSplitWarps);
    gather_split_kernel<<<grid, kSplitWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(*a);
  }
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}
