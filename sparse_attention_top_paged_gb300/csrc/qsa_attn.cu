// qsa_attn.cu — QSA prefill attention over the selected blocks plus the
// incomplete tail ("metrale_model_layers/layers/ops/qsa.rs", qsa_prefill_attn).
//
// Row r sits at position p = first_pos + r; the blocks of `ratio` tokens
// complete by then are b < (p + 1) / ratio. For each (row, query head h) one
// softmax runs over every token of each selected block b = lists[r][i] that is
// complete (others are skipped) and over the tail tokens
// ((p + 1) / ratio) * ratio .. p, with K and V of kv head h / (nq / nkv) read
// through the page table; attn_out[r][h] is the softmax-weighted sum of V.
// With 2, 4 or 8 query heads per kv head and hd <= 128, one CTA per
// (row, kv head) serves the whole group (qsa_prefill_attn_group_kernel);
// otherwise one CTA of 8 warps per (row, head), the page's launch shape: each warp
// keeps an online-softmax partial (reference max, running sum, hd accumulators,
// hd / 32 per lane) over its share of the tokens, one token per step (a
// vector of K and V per lane, a warp sum for the score); the partials are
// merged at the end. (Four tokens per step raised the registers to 76 at
// hd = 128 and ran 23 % slower: fewer resident warps hide less latency.)
#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kAttnWarps = 8;
// Online softmax with a lazy reference maximum: the exponentials are taken
// against a running reference m that moves only when a score exceeds it by
// more than kLazyMax, so the accumulators are rescaled on few tokens and each
// weight exp(s - m) stays below e^kLazyMax (no f32 overflow). Any reference
// gives the same softmax; the partials are merged against their own m.
constexpr float kLazyMax = 8.0f;

template <int HPL>  // head dims per lane (hd = 32 * HPL)
__global__ void __launch_bounds__(kAttnWarps * 32)
    qsa_prefill_attn_kernel(const float *__restrict__ q, const uint16_t *__restrict__ kc,
                            const uint16_t *__restrict__ vc, const int32_t *__restrict__ table, int n_pages, int P,
                            const int32_t *__restrict__ lists, float *__restrict__ out, uint32_t first_pos,
                            uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq, uint32_t nkv,
                            float inv_sqrt_d, int32_t *dev_status) {
  constexpr int hd = 32 * HPL;
  __shared__ float part[kAttnWarps][hd];
  __shared__ float pm[kAttnWarps], pl[kAttnWarps];
  const int r = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long p = static_cast<long long>(first_pos) + r;
  const int kvh = static_cast<int>(h / (nq / nkv));
  float qv[HPL], acc[HPL];
#pragma unroll
  for (int j = 0; j < HPL; ++j) {
    qv[j] = q[(static_cast<long long>(r) * nq + h) * hd + lane * HPL + j] * inv_sqrt_d;
    acc[j] = 0.0f;
  }
  float m = -INFINITY, l = 0.0f;
  bool bad = false;

  auto bf16 = [](uint32_t bits16) { return __uint_as_float(bits16 << 16); };
  auto load = [&](const uint16_t *base, long long off, float (&x)[HPL]) {
    if constexpr (HPL == 2) {
      const uint32_t v = *reinterpret_cast<const uint32_t *>(base + off);
      x[0] = bf16(v & 0xFFFFu); x[1] = bf16(v >> 16);
    } else {
#pragma unroll
      for (int j = 0; j < HPL; j += 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(base + off + j);
        x[j] = bf16(v.x & 0xFFFFu); x[j + 1] = bf16(v.x >> 16);
        x[j + 2] = bf16(v.y & 0xFFFFu); x[j + 3] = bf16(v.y >> 16);
      }
    }
  };
  auto token = [&](long long pos) {
    const long long pg = pos / block_size;
    const int page = pg < n_pages ? table[pg] : -1;
    if (page < 0 || page >= P) {   // warp-uniform: the whole warp handles this token
      bad = true;
      return;
    }
    const long long off = ((static_cast<long long>(page) * block_size + pos % block_size) * nkv + kvh) * hd +
                          lane * HPL;
    float kx[HPL], vx[HPL];
    load(kc, off, kx);
    load(vc, off, vx);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < HPL; ++j) s = fmaf(qv[j], kx[j], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (s > m + kLazyMax) {               // warp-uniform: rescale to the new reference maximum
      const float corr = expf(m - s);     // 0 for the first token (m = -inf)
      l *= corr;
#pragma unroll
      for (int j = 0; j < HPL; ++j) acc[j] *= corr;
      m = s;
    }
    const float e = expf(s - m);          // at most e^kLazyMax
    l += e;
#pragma unroll
    for (int j = 0; j < HPL; ++j) acc[j] = fmaf(e, vx[j], acc[j]);
  };

  const long long ncomp = (p + 1) / ratio;
  for (uint32_t i = warp; i < topk; i += kAttnWarps) {
    const long long b = lists[static_cast<long long>(r) * topk + i];
    if (b < 0 || b >= ncomp) continue;
    for (uint32_t t = 0; t < ratio; ++t) token(b * ratio + t);
  }
  for (long long pos = ncomp * ratio + warp; pos <= p; pos += kAttnWarps) token(pos);

#pragma unroll
  for (int j = 0; j < HPL; ++j) part[warp][lane * HPL + j] = acc[j];
  if (lane == 0) {
    pm[warp] = m;
    pl[warp] = l;
    if (bad && dev_status) atomicOr(dev_status, IDX_STATUS_BAD_BLOCK);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < hd; d += kAttnWarps * 32) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, pm[w]);
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        if (pm[w] == -INFINITY) continue;   // a warp that saw no token
        const float c = expf(pm[w] - M);
        L = fmaf(pl[w], c, L);
        o = fmaf(part[w][d], c, o);
      }
    }
    out[(static_cast<long long>(r) * nq + h) * hd + d] = L > 0.0f ? o / L : 0.0f;
  }
}

// The same attention with one CTA per (row, kv head) covering the G query
// heads of the group: each K and V row is loaded once for all G heads. The G
// partial dot products of a token are reduced across the warp in halving
// steps (lanes keep half the heads at each step: 2G-1 shuffles instead of
// 5G), then each head's score is broadcast from the lane that holds it.
template <int HPL, int G>
__global__ void __launch_bounds__(kAttnWarps * 32)
    qsa_prefill_attn_group_kernel(const float *__restrict__ q, const uint16_t *__restrict__ kc,
                                  const uint16_t *__restrict__ vc, const int32_t *__restrict__ table, int n_pages,
                                  int P, const int32_t *__restrict__ lists, float *__restrict__ out,
                                  uint32_t first_pos, uint32_t topk, uint32_t ratio, uint32_t block_size,
                                  uint32_t nq, uint32_t nkv, float inv_sqrt_d, int32_t *dev_status) {
  constexpr int hd = 32 * HPL;
  constexpr int kLogG = G == 8 ? 3 : (G == 4 ? 2 : 1);
  __shared__ float part[kAttnWarps][G][hd];
  __shared__ float pm[kAttnWarps][G], pl[kAttnWarps][G];
  const int r = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long p = static_cast<long long>(first_pos) + r;
  float qv[G][HPL], acc[G][HPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int h = kvh * G + g;
#pragma unroll
    for (int j = 0; j < HPL; ++j) {
      qv[g][j] = q[(static_cast<long long>(r) * nq + h) * hd + lane * HPL + j] * inv_sqrt_d;
      acc[g][j] = 0.0f;
    }
  }
  // The softmax state of head lane >> (5 - kLogG), kept by the lanes that
  // hold that head's scores: the reference maximum and the running sum.
  float m = -INFINITY, l = 0.0f;
  bool bad = false;

  auto bf16 = [](uint32_t bits16) { return __uint_as_float(bits16 << 16); };
  // A token's K and V words for this lane (HPL bf16 values each), fetched one
  // token ahead of their use so the next token's loads overlap this one's math.
  struct Raw {
    uint32_t k[HPL / 2], v[HPL / 2];
    bool ok;
  };
  auto fetch = [&](long long pos, Raw &x) {
    const long long pg = pos / block_size;
    const int page = pg < n_pages ? table[pg] : -1;
    x.ok = page >= 0 && page < P;   // warp-uniform
    if (!x.ok) return;
    const long long off = ((static_cast<long long>(page) * block_size + pos % block_size) * nkv + kvh) * hd +
                          lane * HPL;
#pragma unroll
    for (int j = 0; j < HPL / 2; j += 2) {
      if constexpr (HPL == 2) {
        x.k[j] = *reinterpret_cast<const uint32_t *>(kc + off);
        x.v[j] = *reinterpret_cast<const uint32_t *>(vc + off);
      } else {
        const uint2 kk = *reinterpret_cast<const uint2 *>(kc + off + 2 * j);
        const uint2 vv = *reinterpret_cast<const uint2 *>(vc + off + 2 * j);
        x.k[j] = kk.x; x.k[j + 1] = kk.y;
        x.v[j] = vv.x; x.v[j + 1] = vv.y;
      }
    }
  };
  auto token = [&](const Raw &x) {
    if (!x.ok) {
      bad = true;
      return;
    }
    float kx[HPL], vx[HPL];
#pragma unroll
    for (int j = 0; j < HPL / 2; ++j) {
      kx[2 * j] = bf16(x.k[j] & 0xFFFFu); kx[2 * j + 1] = bf16(x.k[j] >> 16);
      vx[2 * j] = bf16(x.v[j] & 0xFFFFu); vx[2 * j + 1] = bf16(x.v[j] >> 16);
    }
    float v[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float d = 0.0f;
#pragma unroll
      for (int j = 0; j < HPL; ++j) d = fmaf(qv[g][j], kx[j], d);
      v[g] = d;
    }
    // halving steps over lane bits 4, 3, ...: the upper half of the lanes keeps
    // the upper half of the remaining heads; then plain sums over the rest
#pragma unroll
    for (int st = 0; st < kLogG; ++st) {
      const int o = 16 >> st, half = G >> (st + 1);
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
      }
    }
#pragma unroll
    for (int o = 16 >> kLogG; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
    // lane l now holds the score of head l >> (5 - kLogG)
    const float s = v[0];
    const bool grow = s > m + kLazyMax;
    if (__any_sync(0xFFFFFFFFu, grow)) {   // some head's reference maximum moves up: rescale
      const float m_new = grow ? s : m;
      const float corr = expf(m - m_new);  // 0 on a head's first token, 1 where nothing moved
      l *= corr;
      m = m_new;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float cg = __shfl_sync(0xFFFFFFFFu, corr, g << (5 - kLogG));
#pragma unroll
        for (int j = 0; j < HPL; ++j) acc[g][j] *= cg;
      }
    }
    const float e = expf(s - m);           // at most e^kLazyMax
    l += e;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float eg = __shfl_sync(0xFFFFFFFFu, e, g << (5 - kLogG));
#pragma unroll
      for (int j = 0; j < HPL; ++j) acc[g][j] = fmaf(eg, vx[j], acc[g][j]);
    }
  };

  const long long ncomp = (p + 1) / ratio;
  Raw cur{}, nxt{};
  for (uint32_t i = warp; i < topk; i += kAttnWarps) {
    const long long b = lists[static_cast<long long>(r) * topk + i];
    if (b < 0 || b >= ncomp) continue;
    fetch(b * ratio, cur);
    for (uint32_t t = 0; t < ratio; ++t) {
      if (t + 1 < ratio) fetch(b * ratio + t + 1, nxt);
      token(cur);
      cur = nxt;
    }
  }
  const long long tail0 = ncomp * ratio + warp;
  if (tail0 <= p) fetch(tail0, cur);
  for (long long pos = tail0; pos <= p; pos += kAttnWarps) {
    if (pos + kAttnWarps <= p) fetch(pos + kAttnWarps, nxt);
    token(cur);
    cur = nxt;
  }

#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int j = 0; j < HPL; ++j) part[warp][g][lane * HPL + j] = acc[g][j];
  }
  if ((lane & ((32 >> kLogG) - 1)) == 0) {   // the first lane of each head
    pm[warp][lane >> (5 - kLogG)] = m;
    pl[warp][lane >> (5 - kLogG)] = l;
  }
  if (lane == 0 && bad && dev_status) atomicOr(dev_status, IDX_STATUS_BAD_BLOCK);
  __syncthreads();
  for (int x = threadIdx.x; x < G * hd; x += kAttnWarps * 32) {
    const int g = x / hd, d = x % hd;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, pm[w][g]);
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        if (pm[w][g] == -INFINITY) continue;
        const float c = expf(pm[w][g] - M);
        L = fmaf(pl[w][g], c, L);
        o = fmaf(part[w][g][d], c, o);
      }
    }
    out[(static_cast<long long>(r) * nq + kvh * G + g) * hd + d] = L > 0.0f ? o / L : 0.0f;
  }
}

bool aligned_to(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace
}  // namespace idx

extern "C" idx_status_t idx_qsa_prefill_attn(const float *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                             const int32_t *block_table, int32_t n_pages, int32_t P,
                                             const int32_t *lists, float *attn_out, uint32_t rows,
                                             uint32_t first_pos, uint32_t topk, uint32_t ratio,
                                             uint32_t block_size, uint32_t nq, uint32_t nkv, uint32_t hd,
                                             float inv_sqrt_d, int32_t *dev_status, idx_stream_t stream) {
  using namespace idx;
  if (hd != 64 && hd != 128 && hd != 256) return IDX_ERR_INVALID_ARG;
  if (nkv == 0 || nq % nkv != 0 || ratio == 0 || block_size == 0 || n_pages < 1 || P < 1)
    return IDX_ERR_INVALID_ARG;
  if (rows == 0 || nq == 0) return IDX_OK;
  if (rows > 0x7FFFFFFFu || nq > 65535u) return IDX_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_table || !attn_out || (topk > 0 && !lists)) return IDX_ERR_INVALID_ARG;
  if (!aligned_to(q, 4) || !aligned_to(k_cache, 8) || !aligned_to(v_cache, 8) || !aligned_to(block_table, 4) ||
      (lists && !aligned_to(lists, 4)) || !aligned_to(attn_out, 4) || (dev_status && !aligned_to(dev_status, 4)))
    return IDX_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t G = nq / nkv;
  if ((G == 2 || G == 4 || G == 8) && (hd == 64 || hd == 128)) {
    const dim3 ggrid(rows, nkv);
#define IDX_ATTN_GROUP(HPL_, G_)                                                                              \
  qsa_prefill_attn_group_kernel<HPL_, G_><<<ggrid, kAttnWarps * 32, 0, s>>>(                                  \
      q, k_cache, v_cache, block_table, n_pages, P, lists, attn_out, first_pos, topk, ratio, block_size, nq, nkv, \
      inv_sqrt_d, dev_status)
    if (hd == 64) {
      if (G == 2) IDX_ATTN_GROUP(2, 2); else if (G == 4) IDX_ATTN_GROUP(2, 4); else IDX_ATTN_GROUP(2, 8);
    } else {
      if (G == 2) IDX_ATTN_GROUP(4, 2); else if (G == 4) IDX_ATTN_GROUP(4, 4); else IDX_ATTN_GROUP(4, 8);
    }
#undef IDX_ATTN_GROUP
    return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
  }
  const dim3 grid(rows, nq);
  if (hd == 64)
    qsa_prefill_attn_kernel<2><<<grid, kAttnWarps * 32, 0, s>>>(q, k_cache, v_cache, block_table, n_pages, P, lists,
                                                                attn_out, first_pos, topk, ratio, block_size, nq,
                                                                nkv, inv_sqrt_d, dev_status);
  else if (hd == 128)
    qsa_prefill_attn_kernel<4><<<grid, kAttnWarps * 32, 0, s>>>(q, k_cache, v_cache, block_table, n_pages, P, lists,
                                                                attn_out, first_pos, topk, ratio, block_size, nq,
                                                                nkv, inv_sqrt_d, dev_status);
  else
    qsa_prefill_attn_kernel<8><<<grid, kAttnWarps * 32, 0, s>>>(q, k_cache, v_cache, block_table, n_pages, P, lists,
                                                                attn_out, first_pos, topk, ratio, block_size, nq,
                                                                nkv, inv_sqrt_d, dev_status);
  return cudaGetLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}
