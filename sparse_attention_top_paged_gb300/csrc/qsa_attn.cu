// qsa_attn.cu — QSA prefill attention over the selected blocks plus the
// incomplete tail ("metrale_model_layers/layers/ops/qsa.rs", qsa_prefill_attn).
//
// Row r sits at position p = first_pos + r; the blocks of `ratio` tokens
// complete by then are b < (p + 1) / ratio. For each (row, query head h) one
// softmax runs over every token of each selected block b = lists[r][i] that is
// complete (others are skipped) and over the tail tokens
// ((p + 1) / ratio) * ratio .. p, with K and V of kv head h / (nq / nkv) read
// through the page table; attn_out[r][h] is the softmax-weighted sum of V.
// With 1, 2, 4 or 8 query heads per kv head, hd <= 128 and a 16-byte aligned
// K cache, one CTA per (row, kv head) serves the whole group over 32-token
// tiles (qsa_prefill_attn_tile_kernel: lane per token for the scores, lane
// per dimension for the V sum). Otherwise one CTA of 8 warps per (row, head),
// the page's launch shape: each warp keeps an online-softmax partial
// (reference max, running sum, hd accumulators, hd / 32 per lane) over its
// share of the tokens, one token per step (a vector of K and V per lane, a
// warp sum for the score); the partials are merged at the end.
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

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared-memory bytes of qsa_prefill_attn_tile_kernel<HD, G>.
template <int HD, int G>
constexpr size_t tile_smem_bytes() {
  return static_cast<size_t>(kAttnWarps) * 32 * (HD * 2 + 16)   // staged K rows (padded)
         + G * HD * 4                                          // scaled q of the group
         + kAttnWarps * 32 * G * 4                             // the tile's weights
         + 2 * kAttnWarps * 32 * 8                             // row offsets of this tile and the next
         + 2 * kAttnWarps * G * 4;                             // per-warp maxima and sums
}

// The same attention over 32-token tiles, one CTA of 8 warps per (row, kv
// head) serving its G query heads (G = 1, 2, 4 or 8; hd = 64 or 128). For the
// scores lane t owns token t of the warp's tile: the tile's K rows are staged
// into shared memory with coalesced asynchronous copies (rows padded by 16
// bytes so that lanes reading the same chunk of different rows hit distinct
// banks), and each lane forms its token's G dot products against q broadcast
// from shared memory: no per-token shuffle reduction. The weighted V sum then
// gives each lane hd / 32 dimensions and walks the tile's tokens. Once the scores are formed, the same staging rows receive
// the tile's V rows (one asynchronous copy per tile, not a load per token),
// while the next tile's offsets are looked up and the softmax runs. Tokens
// are numbered list-major (token t of selected block i is i * ratio + t,
// blocks that are not complete masked out), then the tail.
template <int HD, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, 2)
    qsa_prefill_attn_tile_kernel(const float *__restrict__ q, const uint16_t *__restrict__ kc,
                                 const uint16_t *__restrict__ vc, const int32_t *__restrict__ table, int n_pages,
                                 int P, const int32_t *__restrict__ lists, float *__restrict__ out,
                                 uint32_t first_pos, uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq,
                                 uint32_t nkv, float inv_sqrt_d, int32_t *dev_status) {
  constexpr int HPL = HD / 32;        // dimensions per lane in the V sum
  constexpr int NC = HD / 8;          // 16-byte chunks of a K row
  constexpr int ROWB = HD * 2 + 16;   // staged row stride in bytes
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char *kbuf = smem;
  float *qs = reinterpret_cast<float *>(smem + static_cast<size_t>(kAttnWarps) * 32 * ROWB);
  float *ps = qs + G * HD;
  long long *roff = reinterpret_cast<long long *>(ps + kAttnWarps * 32 * G);
  float *pm = reinterpret_cast<float *>(roff + 2 * kAttnWarps * 32);
  float *pl = pm + kAttnWarps * G;
  float *part = reinterpret_cast<float *>(smem);   // [warp][G][HD] after the tiles: aliases the staged rows
  static_assert(kAttnWarps * G * HD * 4 <= kAttnWarps * 32 * ROWB, "merge buffer fits the staging area");

  const int r = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long p = static_cast<long long>(first_pos) + r;
  for (int x = threadIdx.x; x < G * HD; x += kAttnWarps * 32)
    qs[x] = q[(static_cast<long long>(r) * nq + static_cast<long long>(kvh) * G + x / HD) * HD + x % HD] * inv_sqrt_d;
  __syncthreads();

  const long long ncomp = (p + 1) / ratio;
  const long long n_list = static_cast<long long>(topk) * ratio;
  const long long tail0 = ncomp * ratio;
  const long long n_virt = n_list + (p + 1 - tail0);
  unsigned char *kw = kbuf + static_cast<size_t>(warp) * 32 * ROWB;
  float *pw = ps + warp * 32 * G;
  long long *ow2 = roff + warp * 64;   // [2][32]: this tile's and the next tile's row offsets
  float acc[G][HPL], m[G], l[G];   // m: the head's reference maximum (warp-uniform); l: this lane's share of the sum
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int j = 0; j < HPL; ++j) acc[g][j] = 0.0f;
  }
  bool bad = false;

  // The K/V element offset of this lane's token of the tile starting at
  // virtual token `base`, or -1 (no token, or its page is missing).
  auto token_offset = [&](long long base) -> long long {
    const long long v = base + lane;
    long long pos = -1;
    if (v < n_list) {
      const long long b = lists[static_cast<long long>(r) * topk + v / ratio];
      if (b >= 0 && b < ncomp) pos = b * ratio + v % ratio;
    } else if (v < n_virt) {
      pos = tail0 + (v - n_list);
    }
    if (pos < 0) return -1;
    const long long pg = pos / block_size;
    const int page = pg < n_pages ? table[pg] : -1;
    if (page < 0 || page >= P) {
      bad = true;
      return -1;
    }
    return ((static_cast<long long>(page) * block_size + pos % block_size) * nkv + kvh) * HD;
  };
  // Copies the K or V rows listed in o[0..31] into the staging rows
  // (consecutive lanes: consecutive chunks of one row) as one asynchronous group.
  auto stage = [&](const uint16_t *cache, const long long *o) {
    for (int x = lane; x < 32 * NC; x += 32) {
      const int t = x / NC, c = x % NC;
      const long long src = o[t];
      if (src >= 0) cp_async16(kw + t * ROWB + c * 16, cache + src + c * 8);
    }
    cp_async_commit();
  };

  long long base = static_cast<long long>(warp) * 32;
  long long off = base < n_virt ? token_offset(base) : -1;
  uint32_t live = __ballot_sync(0xFFFFFFFFu, off >= 0);
  ow2[lane] = off;
  for (int buf = 0; base < n_virt; base += kAttnWarps * 32, buf ^= 1) {
    const long long *ow = ow2 + 32 * buf;
    __syncwarp();
    stage(kc, ow);
    cp_async_wait_all();
    __syncwarp();
    constexpr int NCH = G >= 4 ? 1 : 2;   // dependent chains per head (G >= 4 heads already interleave)
    float sa[NCH][G];
#pragma unroll
    for (int u = 0; u < NCH; ++u)
#pragma unroll
      for (int g = 0; g < G; ++g) sa[u][g] = 0.0f;
    if (off >= 0) {
      const unsigned char *kr = kw + lane * ROWB;
#pragma unroll 2
      for (int c = 0; c < NC; ++c) {
        const uint4 w = *reinterpret_cast<const uint4 *>(kr + c * 16);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        float kx[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kx[2 * e] = __uint_as_float(wv[e] << 16);
          kx[2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4 *>(qs + g * HD + 8 * c);
          const float4 qb = *reinterpret_cast<const float4 *>(qs + g * HD + 8 * c + 4);
          float &a = sa[c % NCH][g];
          a = fmaf(qa.x, kx[0], a); a = fmaf(qa.y, kx[1], a); a = fmaf(qa.z, kx[2], a); a = fmaf(qa.w, kx[3], a);
          a = fmaf(qb.x, kx[4], a); a = fmaf(qb.y, kx[5], a); a = fmaf(qb.z, kx[6], a); a = fmaf(qb.w, kx[7], a);
        }
      }
    }
    __syncwarp();   // every lane has read its K row: the V rows may land
    stage(vc, ow);
    const long long nbase = base + kAttnWarps * 32;
    const long long noff = nbase < n_virt ? token_offset(nbase) : -1;
    const uint32_t nlive = __ballot_sync(0xFFFFFFFFu, noff >= 0);
    ow2[32 * (buf ^ 1) + lane] = noff;
    float ev[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sc = off >= 0 ? (NCH == 2 ? sa[0][g] + sa[NCH - 1][g] : sa[0][g]) : -INFINITY;
      float mt = sc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
      if (mt > m[g] + kLazyMax) {   // warp-uniform: rescale to the new reference maximum
        const float corr = expf(m[g] - mt);
        l[g] *= corr;
#pragma unroll
        for (int j = 0; j < HPL; ++j) acc[g][j] *= corr;
        m[g] = mt;
      }
      ev[g] = off >= 0 ? expf(sc - m[g]) : 0.0f;
      l[g] += ev[g];
    }
    if constexpr (G % 4 == 0) {
#pragma unroll
      for (int g = 0; g < G; g += 4)
        *reinterpret_cast<float4 *>(pw + lane * G + g) = make_float4(ev[g], ev[g + 1], ev[g + 2], ev[g + 3]);
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) pw[lane * G + g] = ev[g];
    }
    cp_async_wait_all();
    __syncwarp();
#pragma unroll 4
    for (int t = 0; t < 32; ++t) {
      if (!((live >> t) & 1u)) continue;
      const unsigned char *vr = kw + t * ROWB + lane * HPL * 2;
      float vx[HPL];
      if constexpr (HPL == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(vr);
        vx[0] = __uint_as_float(w << 16); vx[1] = __uint_as_float(w & 0xFFFF0000u);
      } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(vr);
        vx[0] = __uint_as_float(w.x << 16); vx[1] = __uint_as_float(w.x & 0xFFFF0000u);
        vx[2] = __uint_as_float(w.y << 16); vx[3] = __uint_as_float(w.y & 0xFFFF0000u);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pt = pw[t * G + g];
#pragma unroll
        for (int j = 0; j < HPL; ++j) acc[g][j] = fmaf(pt, vx[j], acc[g][j]);
      }
    }
    off = noff;   // the next tile rewrites pw and kw after the __syncwarp at its top
    live = nlive;
  }

#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l[g] += __shfl_xor_sync(0xFFFFFFFFu, l[g], o);
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && dev_status) atomicOr(dev_status, IDX_STATUS_BAD_BLOCK);
  __syncthreads();   // every warp is done with its staged rows: part reuses them
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int j = 0; j < HPL; ++j) part[(warp * G + g) * HD + lane * HPL + j] = acc[g][j];
    if (lane == 0) {
      pm[warp * G + g] = m[g];
      pl[warp * G + g] = l[g];
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < G * HD; x += kAttnWarps * 32) {
    const int g = x / HD, d = x % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, pm[w * G + g]);
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        if (pm[w * G + g] == -INFINITY) continue;   // a warp that saw no token
        const float c = expf(pm[w * G + g] - M);
        L = fmaf(pl[w * G + g], c, L);
        o = fmaf(part[(w * G + g) * HD + d], c, o);
      }
    }
    out[(static_cast<long long>(r) * nq + static_cast<long long>(kvh) * G + g) * HD + d] = L > 0.0f ? o / L : 0.0f;
  }
}

template <int HD, int G>
cudaError_t launch_tile(dim3 grid, cudaStream_t s, const float *q, const uint16_t *kc, const uint16_t *vc,
                        const int32_t *table, int n_pages, int P, const int32_t *lists, float *out,
                        uint32_t first_pos, uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq,
                        uint32_t nkv, float inv_sqrt_d, int32_t *dev_status) {
  constexpr size_t bytes = tile_smem_bytes<HD, G>();
  static const cudaError_t attr = cudaFuncSetAttribute(qsa_prefill_attn_tile_kernel<HD, G>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(bytes));
  if (attr != cudaSuccess) return attr;
  qsa_prefill_attn_tile_kernel<HD, G><<<grid, kAttnWarps * 32, bytes, s>>>(
      q, kc, vc, table, n_pages, P, lists, out, first_pos, topk, ratio, block_size, nq, nkv, inv_sqrt_d, dev_status);
  return cudaGetLastError();
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
  if ((G == 1 || G == 2 || G == 4 || G == 8) && (hd == 64 || hd == 128) && aligned_to(k_cache, 16)) {
    const dim3 tgrid(rows, nkv);
#define IDX_ATTN_TILE(HD_, G_)                                                                                  \
  launch_tile<HD_, G_>(tgrid, s, q, k_cache, v_cache, block_table, n_pages, P, lists, attn_out, first_pos, topk, \
                       ratio, block_size, nq, nkv, inv_sqrt_d, dev_status)
    cudaError_t e;
    if (hd == 64)
      e = G == 1 ? IDX_ATTN_TILE(64, 1) : G == 2 ? IDX_ATTN_TILE(64, 2) : G == 4 ? IDX_ATTN_TILE(64, 4)
                                                                            : IDX_ATTN_TILE(64, 8);
    else
      e = G == 1 ? IDX_ATTN_TILE(128, 1) : G == 2 ? IDX_ATTN_TILE(128, 2) : G == 4 ? IDX_ATTN_TILE(128, 4)
                                                                              : IDX_ATTN_TILE(128, 8);
#undef IDX_ATTN_TILE
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
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
