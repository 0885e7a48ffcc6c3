// score_simt.cu — CUDA-core scorer: writes every I[t,s] to a score matrix.
//
// The unquantised (F32) key path of idx_score_topk, and a second, independent
// GPU implementation of the NVFP4 scores next to the tensor-core kernel. G
// consecutive lanes own one key: each resolves the key's row through the
// block table, decodes the whole row into registers once, then runs heads
// hg, hg + G, ... against q held in shared memory, and the G partial sums
// meet in a shuffle reduction (eq. 16 of "indexer_score_topk.cu":
// I = sum_h w_h * ReLU(q_h . K_s); its main loop also decodes each key once
// per query, but serially per thread over strided keys). G = 1 when there
// are keys enough to fill the GPU, else 8 (e.g. one decode query over a few
// hundred pooled blocks), so that short rows still spread over many SMs.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kSimtThreads = 64;

__constant__ float kE2m1Lut[16] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f,
                                   -0.0f, -0.5f, -1.0f, -1.5f, -2.0f, -3.0f, -4.0f, -6.0f};

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
  return __half2float(__half(h));
}

template <int D, bool F32, int G>
__global__ void __launch_bounds__(kSimtThreads) score_simt_kernel(ScoreParams p, float *scores,
                                                                  long long ld) {
  constexpr int QS = G > 1 ? D + 4 : D;   // q row stride: G lanes read G heads on distinct banks
  extern __shared__ float smem[];
  float *q_s = smem;             // [H][QS]
  float *w_s = smem + p.H * QS;  // [H]
  const int t = blockIdx.y;
  const int L = p.valid_lens[t];
  if (L < 0 || static_cast<long long>(L) > static_cast<long long>(p.max_lb) * p.epb) return;
  const int s0 = blockIdx.x * (kSimtThreads / G);
  if (s0 >= L) return;

  const float *qt = p.q + static_cast<long long>(t) * p.H * D;
  for (int i = threadIdx.x; i < p.H * D / 4; i += kSimtThreads) {
    const int h = (4 * i) / D, d = (4 * i) % D;
    *reinterpret_cast<float4 *>(q_s + h * QS + d) = reinterpret_cast<const float4 *>(qt)[i];
  }
  for (int h = threadIdx.x; h < p.H; h += kSimtThreads) w_s[h] = p.w[static_cast<long long>(t) * p.H + h];
  __syncthreads();

  const int hg = threadIdx.x % G;   // this lane's first head
  const int s = s0 + threadIdx.x / G;
  bool bad = false;
  float I = -INFINITY;   // a bad block: -inf from every lane of the key
  if (s < L) {
    const int lb = s / p.epb, slot = s % p.epb;
    const int phys = p.block_table[static_cast<long long>(t) * p.bt_stride + lb];
    if (phys < 0 || phys >= p.P) {
      bad = true;
    } else {
      const long long row = static_cast<long long>(phys) * p.epb + slot;
      float k[D];
      if constexpr (F32) {
        const float4 *src = reinterpret_cast<const float4 *>(p.keys_f32 + row * D);
#pragma unroll
        for (int i = 0; i < D / 4; ++i) {
          const float4 v = src[i];
          k[4 * i] = v.x; k[4 * i + 1] = v.y; k[4 * i + 2] = v.z; k[4 * i + 3] = v.w;
        }
      } else {
        const float g = p.key_gscale[phys];
        const uint4 *src = reinterpret_cast<const uint4 *>(p.keys_fp4 + row * (D / 2));
        const uint8_t *sc = p.key_scale + row * (D / 16);
#pragma unroll
        for (int grp = 0; grp < D / 16; ++grp) {
          const float gs = e4m3_to_float(sc[grp]) * g;
          const uint4 raw4 = src[grp / 2];
          const uint32_t wlo = (grp & 1) ? raw4.z : raw4.x;
          const uint32_t whi = (grp & 1) ? raw4.w : raw4.y;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const uint32_t byte = ((b < 4 ? wlo : whi) >> (8 * (b & 3))) & 0xFFu;
            k[grp * 16 + 2 * b] = kE2m1Lut[byte & 0xFu] * gs;
            k[grp * 16 + 2 * b + 1] = kE2m1Lut[byte >> 4] * gs;
          }
        }
      }
      I = 0.0f;
      for (int h = hg; h < p.H; h += G) {
        const float *qh = q_s + h * QS;
        float dot0 = 0.0f, dot1 = 0.0f, dot2 = 0.0f, dot3 = 0.0f;   // four independent chains
#pragma unroll
        for (int d = 0; d < D; d += 4) {
          dot0 = fmaf(qh[d], k[d], dot0);
          dot1 = fmaf(qh[d + 1], k[d + 1], dot1);
          dot2 = fmaf(qh[d + 2], k[d + 2], dot2);
          dot3 = fmaf(qh[d + 3], k[d + 3], dot3);
        }
        const float dot = (dot0 + dot1) + (dot2 + dot3);
        I = fmaf(w_s[h], fmaxf(dot, 0.0f), I);
      }
    }
  }
  // the G lanes of a key are consecutive and all reach here (a key past L, or
  // with a bad block, is the same for all of them)
#pragma unroll
  for (int o = 1; o < G; o <<= 1) I += __shfl_xor_sync(0xFFFFFFFFu, I, o);
  if (s < L && hg == 0 && IDX_IN_BOUNDS(t < p.T && s < ld, p.dev_status)) scores[static_cast<long long>(t) * ld + s] = I;
  if (__any_sync(0xFFFFFFFFu, bad) && lane_id() == 0 && p.dev_status)
    atomicOr(p.dev_status, IDX_STATUS_BAD_BLOCK);
}

template <int D, bool F32, int G>
cudaError_t launch_g(const ScoreParams &p, float *scores, long long ld, cudaStream_t stream) {
  constexpr int QS = G > 1 ? D + 4 : D;
  const size_t smem = static_cast<size_t>(p.H) * QS * 4 + static_cast<size_t>(p.H) * 4;
  auto kern = score_simt_kernel<D, F32, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long max_len = static_cast<long long>(p.max_lb) * p.epb;
  constexpr int keys_per_cta = kSimtThreads / G;
  dim3 grid(static_cast<unsigned>((max_len + keys_per_cta - 1) / keys_per_cta), p.T);
  kern<<<grid, kSimtThreads, smem, stream>>>(p, scores, ld);
  return cudaGetLastError();
}

// One lane per key when the keys fill every SM several times over; else 8
// lanes per key (heads split eight ways).
template <int D, bool F32>
cudaError_t launch_one(const ScoreParams &p, float *scores, long long ld, cudaStream_t stream) {
  const long long keys = static_cast<long long>(p.T) * p.max_lb * p.epb;
  const int sms = device_sm_count();
  if (p.H % 8 == 0 && keys < 4LL * kSimtThreads * (sms > 0 ? sms : 148))
    return launch_g<D, F32, 8>(p, scores, ld, stream);
  return launch_g<D, F32, 1>(p, scores, ld, stream);
}

}  // namespace

cudaError_t launch_score_simt(const ScoreParams &p, bool f32_keys, float *scores, long long ld,
                              cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  if (f32_keys) {
    if (p.D == 64) return launch_one<64, true>(p, scores, ld, stream);
    return launch_one<128, true>(p, scores, ld, stream);
  }
  return launch_one<128, false>(p, scores, ld, stream);
}

}  // namespace idx
