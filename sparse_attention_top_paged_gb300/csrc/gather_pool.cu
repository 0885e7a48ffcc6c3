// gather_pool.cu — the selected-row K/V gather, QSA block-key pooling, the
// block -> position expansion for the gather, and valid lengths from block
// counts.
#include <climits>

#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

// ---------------------------------------------------------------- gather ----
// qsa.rs, qsa_gather: slot i of the dense output holds position sel[i]; the
// row is found through the block table (commit c2f705a's gather_kv resolves
// rows the same way). One warp copies one row in 16-byte vectors.
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) gather_kv_kernel(idx_gather_kv_args a) {
  const long long r = static_cast<long long>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  const long long n_rows = static_cast<long long>(a.T) * a.n_sel;
  if (r >= n_rows) return;
  const int t = static_cast<int>(r / a.n_sel);
  const int pos = a.sel[r];
  long long src_row = -1;
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
        src_row = static_cast<long long>(phys) * a.block_size + pos % a.block_size;
    }
  }
  if (err && lane_id() == 0 && a.dev_status) atomicOr(a.dev_status, err);
  if (src_row >= 0 && !IDX_IN_BOUNDS(src_row < static_cast<long long>(a.P) * a.block_size, a.dev_status)) src_row = -1;
  const long long nvec = a.row_bytes / 16;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint4 *ks = static_cast<const uint4 *>(a.k_cache) + (src_row >= 0 ? src_row : 0) * nvec;
  const uint4 *vs = a.v_cache ? static_cast<const uint4 *>(a.v_cache) + (src_row >= 0 ? src_row : 0) * nvec : nullptr;
  uint4 *kd = static_cast<uint4 *>(a.k_out) + r * nvec;
  uint4 *vd = a.v_cache ? static_cast<uint4 *>(a.v_out) + r * nvec : nullptr;
  // two 16-byte pieces of the K row and of the V row a lane at a time, all four
  // loads issued before any store (a store could alias a later load, so the
  // compiler would not move the load ahead of it)
  for (long long c0 = lane_id(); c0 < nvec; c0 += 64) {
    const long long c1 = c0 + 32;
    const bool has1 = c1 < nvec;
    const uint4 k0 = src_row >= 0 ? __ldg(ks + c0) : zero;
    const uint4 k1 = (src_row >= 0 && has1) ? __ldg(ks + c1) : zero;
    uint4 v0 = zero, v1 = zero;
    if (vs != nullptr && src_row >= 0) {
      v0 = __ldg(vs + c0);
      if (has1) v1 = __ldg(vs + c1);
    }
    __stcs(kd + c0, k0);
    if (has1) __stcs(kd + c1, k1);
    if (vd != nullptr) {
      __stcs(vd + c0, v0);
      if (has1) __stcs(vd + c1, v1);
    }
  }
}

// ------------------------------------------------------------ block pool ----
// qsa.rs, qsa_block_pool: per block, the mean of `ratio` raw keys, RMSNorm
// scaled by (1 + w), then rope on the first `rot` dimensions at the block's
// first token position. One CTA per block, one thread per dimension (the
// page's launch shape: grid n_new, block hd). Rope pairs d with d + rot/2.
// The frequencies theta^(-2i/rot) come from the host in double precision, the
// angle pos * freq is formed in double and reduced to [-pi, pi] in double,
// and only the sine and cosine of the reduced angle are taken in single
// precision (double-precision trigonometry per thread cost more than the rest
// of the kernel).
constexpr int kMaxRopeFreqs = 512;  // rot <= hd <= 1024
struct RopeFreqs {
  double f[kMaxRopeFreqs];
};

// One row of hd values (the mean of `nrow` bf16 rows `stride` elements apart)
// -> RMSNorm scaled by (1 + w) -> rope at `pos` -> dst. One thread per
// dimension; `sm` holds hd + 32 floats. Shared by the block pooling and the
// query preparation, which differ only in where their rows come from.
__device__ __forceinline__ void norm_rope_row(const uint16_t *__restrict__ src, long long stride, uint32_t nrow,
                                              const float *__restrict__ w, float *__restrict__ dst, uint32_t hd,
                                              uint32_t rot, double pos, float eps, const RopeFreqs &rf, float *sm) {
  float *y_s = sm;
  float *red = sm + hd;
  const uint32_t d = threadIdx.x;
  float m = 0.0f;
  for (uint32_t r = 0; r < nrow; ++r) {
    const uint32_t bits = src[static_cast<long long>(r) * stride + d];
    m += __uint_as_float(bits << 16);
  }
  m = m / static_cast<float>(nrow);
  float sq = m * m;
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
  if (lane_id() == 0) red[d >> 5] = sq;
  __syncthreads();
  if (d < 32) {
    float v = (d < (hd + 31) / 32) ? red[d] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (d == 0) red[0] = v;
  }
  __syncthreads();
  const float inv_rms = rsqrtf(red[0] / static_cast<float>(hd) + eps);
  const float y = m * inv_rms * (1.0f + w[d]);
  y_s[d] = y;
  __syncthreads();
  float o = y;
  const uint32_t half = rot / 2;
  if (d < rot) {
    const uint32_t i = d < half ? d : d - half;
    const double ang = pos * rf.f[i];
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    const double turns = rint(ang * (1.0 / kTwoPi));
    const float rd = static_cast<float>(fma(-turns, kTwoPi, ang));
    float s, c;
    sincosf(rd, &s, &c);
    if (d < half)
      o = y * c - y_s[d + half] * s;
    else
      o = y * c + y_s[d - half] * s;
  }
  dst[d] = o;
}

__global__ void block_pool_kernel(const uint16_t *__restrict__ raw, const float *__restrict__ w,
                                  float *__restrict__ out, uint32_t first_block, uint32_t ratio,
                                  uint32_t hd, uint32_t rot, float eps, const __grid_constant__ RopeFreqs rf) {
  extern __shared__ float sm[];  // [hd] pooled-normalised values, then [32] partial sums
  const uint32_t b = first_block + blockIdx.x;
  norm_rope_row(raw + static_cast<long long>(b) * ratio * hd, hd, ratio, w, out + static_cast<long long>(b) * hd,
                hd, rot, static_cast<double>(b) * ratio, eps, rf, sm);
}

// qsa.rs, qsa_qprep / qsa_qprep_rows: row r, head h of the indexer
// projection (q of head h at columns h*hd of a row of width qkw) -> RMSNorm
// scaled by (1 + w) -> rope at position first_pos + r. Grid (rows, n_heads),
// one thread per dimension, as on the page.
__global__ void qsa_qprep_kernel(const uint16_t *__restrict__ qk, const float *__restrict__ w,
                                 float *__restrict__ q_out, uint32_t first_pos, uint32_t qkw, uint32_t n_heads,
                                 uint32_t hd, uint32_t rot, float eps, const __grid_constant__ RopeFreqs rf) {
  extern __shared__ float sm[];
  const uint32_t r = blockIdx.x, h = blockIdx.y;
  norm_rope_row(qk + static_cast<long long>(r) * qkw + static_cast<long long>(h) * hd, 0, 1, w,
                q_out + (static_cast<long long>(r) * n_heads + h) * hd, hd, rot,
                static_cast<double>(first_pos) + r, eps, rf, sm);
}

// --------------------------------------------------------- expand blocks ----
// Selected block ids -> ascending token positions for the gather.
constexpr int kExpandThreads = 256;

__global__ void __launch_bounds__(kExpandThreads) expand_blocks_kernel(const int32_t *blocks, int n_blocks,
                                                                       int ratio, int32_t *positions) {
  extern __shared__ int32_t ids[];   // m sorted ids, then (rank path) the n_blocks ids as read
  const int t = blockIdx.x;
  int m = 1;
  while (m < n_blocks) m <<= 1;
  if (n_blocks <= kExpandThreads) {
    // one thread per id: its place in ascending order is the number of smaller
    // ids, plus the equal ones read before it (two barriers instead of a network)
    int32_t *in = ids + m;
    const int i = threadIdx.x;
    int32_t v = INT_MAX;   // (invalid ids sort last)
    if (i < n_blocks) {
      const int32_t b = blocks[static_cast<long long>(t) * n_blocks + i];
      if (b >= 0) v = b;
      in[i] = v;
    }
    __syncthreads();
    if (i < n_blocks) {
      int rank = 0;
      for (int j = 0; j < n_blocks; ++j) {
        const int32_t u = in[j];
        rank += (u < v || (u == v && j < i)) ? 1 : 0;
      }
      ids[rank] = v;
    }
    __syncthreads();
  } else {
    for (int i = threadIdx.x; i < m; i += kExpandThreads) {
      int32_t v = INT_MAX;
      if (i < n_blocks) {
        const int32_t b = blocks[static_cast<long long>(t) * n_blocks + i];
        if (b >= 0) v = b;
      }
      ids[i] = v;
    }
    __syncthreads();
    for (int size = 2; size <= m; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < (m >> 1); i += kExpandThreads) {
          const int lo = ((i & ~(stride - 1)) << 1) | (i & (stride - 1)), hi = lo + stride;
          const bool asc = (lo & size) == 0;
          const int32_t a = ids[lo], c = ids[hi];
          if ((a > c) == asc) {
            ids[lo] = c;
            ids[hi] = a;
          }
        }
        __syncthreads();
      }
    }
  }
  const long long n_out = static_cast<long long>(n_blocks) * ratio;
  for (long long i = threadIdx.x; i < n_out; i += kExpandThreads) {
    const int32_t b = ids[i / ratio];
    positions[static_cast<long long>(t) * n_out + i] =
        (b == INT_MAX) ? -1 : static_cast<int32_t>(static_cast<long long>(b) * ratio + i % ratio);
  }
}

__global__ void valid_lens_kernel(const int32_t *block_lens, int T, int epb, int32_t *valid_lens) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) valid_lens[t] = block_lens[t] * epb;
}

}  // namespace

cudaError_t launch_gather_kv(const idx_gather_kv_args &a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.T) * a.n_sel;
  if (rows == 0) return cudaSuccess;
  const long long grid = (rows + kGatherWarps - 1) / kGatherWarps;
  gather_kv_kernel<<<static_cast<unsigned>(grid), kGatherWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_block_pool(const uint16_t *raw, const float *w, float *out, uint32_t first_block,
                              uint32_t n_new, uint32_t ratio, uint32_t hd, uint32_t rot, float theta,
                              float eps, cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(hd) + 32) * sizeof(float);
  if (rot / 2 > static_cast<uint32_t>(kMaxRopeFreqs)) return cudaErrorInvalidValue;
  RopeFreqs rf;
  for (uint32_t i = 0; i < rot / 2; ++i)
    rf.f[i] = std::pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(rot));
  block_pool_kernel<<<n_new, hd, smem, stream>>>(raw, w, out, first_block, ratio, hd, rot, eps, rf);
  return cudaGetLastError();
}

cudaError_t launch_qsa_qprep(const uint16_t *qk, const float *w, float *q_out, uint32_t rows, uint32_t first_pos,
                             uint32_t qkw, uint32_t n_heads, uint32_t hd, uint32_t rot, float theta, float eps,
                             cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(hd) + 32) * sizeof(float);
  if (rot / 2 > static_cast<uint32_t>(kMaxRopeFreqs)) return cudaErrorInvalidValue;
  RopeFreqs rf;
  for (uint32_t i = 0; i < rot / 2; ++i)
    rf.f[i] = std::pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(rot));
  qsa_qprep_kernel<<<dim3(rows, n_heads), hd, smem, stream>>>(qk, w, q_out, first_pos, qkw, n_heads, hd, rot, eps,
                                                              rf);
  return cudaGetLastError();
}

cudaError_t launch_expand_blocks(const int32_t *blocks, int T, int n_blocks, int ratio,
                                 int32_t *positions, cudaStream_t stream) {
  if (T == 0 || n_blocks == 0) return cudaSuccess;
  int m = 1;
  while (m < n_blocks) m <<= 1;
  const size_t smem = static_cast<size_t>(n_blocks <= kExpandThreads ? 2 * m : m) * 4;   // (the rank path reads a copy)
  expand_blocks_kernel<<<T, kExpandThreads, smem, stream>>>(blocks, n_blocks, ratio, positions);
  return cudaGetLastError();
}

cudaError_t launch_valid_lens(const int32_t *block_lens, int T, int epb, int32_t *valid_lens,
                              cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  valid_lens_kernel<<<(T + 255) / 256, 256, 0, stream>>>(block_lens, T, epb, valid_lens);
  return cudaGetLastError();
}

}  // namespace idx
