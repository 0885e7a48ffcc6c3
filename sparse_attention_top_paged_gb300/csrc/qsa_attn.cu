// qsa_attn.cu — QSA prefill attention over the selected blocks plus the
// incomplete tail ("metrale_model_layers/layers/ops/qsa.rs", qsa_prefill_attn).
//
// Row r sits at position p = first_pos + r; the blocks of `ratio` tokens
// complete by then are b < (p + 1) / ratio. For each (row, query head h) one
// softmax runs over every token of each selected block b = lists[r][i] that is
// complete (others are skipped) and over the tail tokens
// ((p + 1) / ratio) * ratio .. p, with K and V of kv head h / (nq / nkv) read
// through the page table; attn_out[r][h] is the softmax-weighted sum of V.
// With 1, 2, 4 or 8 query heads per kv head, hd = 128, 16-byte aligned K and V
// caches and 8-byte aligned q, qsa_attn_tc.cu's kernel runs (a persistent
// pipeline over (row, kv head) items in 128-token steps, both contractions on
// tcgen05). With 1, 2, 4 or 8 query heads per kv head otherwise, hd <= 128 and
// 16-byte aligned caches, one CTA per (row, kv head) serves the whole group
// over 32-token tiles
// (qsa_prefill_attn_tile_kernel: both contractions of a tile as warp-level
// mma.sync). Otherwise one CTA of 8 warps per (row, head),
// the page's launch shape: each warp keeps an online-softmax partial
// (reference max, running sum, hd accumulators, hd / 32 per lane) over its
// share of the tokens, one token per step (a vector of K and V per lane, a
// warp sum for the score); the partials are merged at the end.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace idx {

// qsa_attn_tc.cu: the tcgen05 kernel for 1, 2, 4 or 8 query heads per kv head, hd = 128.
bool qsa_attn_tc_supported(const float *q, uint32_t nq, uint32_t nkv, uint32_t hd, const void *kc, const void *vc,
                           uint32_t rows, uint32_t first_pos, uint32_t topk, uint32_t ratio, int P,
                           uint32_t block_size);
cudaError_t launch_qsa_attn_tc(const float *q, const uint16_t *kc, const uint16_t *vc, const int32_t *table,
                               int n_pages, int P, const int32_t *lists, float *out, uint32_t rows, uint32_t first_pos,
                               uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq, uint32_t nkv,
                               float inv_sqrt_d, int32_t *dev_status, cudaStream_t stream);

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

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr) : "memory");
}

// c += a . b on one m16n8k16 tile: a 16x16 bf16 (row-major), b 16x8 bf16
// (column-major), c 16x8 f32.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared-memory bytes of qsa_prefill_attn_tile_kernel<HD, G>.
template <int HD, int G>
constexpr size_t tile_smem_bytes() {
  return static_cast<size_t>(kAttnWarps) * 32 * (HD * 2 + 16)   // staged K, then V, rows (padded)
         + 2 * 8 * (HD + 8) * 2                                // scaled q, bf16 hi and lo rows (8 heads)
         + kAttnWarps * 2 * 8 * 40 * 2                         // the tile's weights, bf16 hi and lo [head][token]
         + 2 * kAttnWarps * 32 * 8                             // row offsets of this tile and the next
         + 2 * kAttnWarps * G * 4;                             // per-warp maxima and sums
}

// The same attention over 32-token tiles, one CTA of 8 warps per (row, kv
// head) serving its G query heads (G = 1, 2, 4 or 8; hd = 64 or 128), both
// contractions on the tensor cores (mma.sync m16n8k16, bf16 in, f32
// accumulate):
//   scores  S[32 tokens x 8 heads] = K_tile . q^T. The tile's K rows are
//           staged into shared memory by coalesced asynchronous copies (rows
//           padded by 16 bytes, so ldmatrix reads them without bank
//           conflicts). K is bf16 already; q * inv_sqrt_d is split into a
//           bf16 high part and a bf16 low part (the rounding residual), two
//           MMAs, so q keeps about 17 significant bits.
//   V sum   O^T[hd x 8 heads] += V_tile^T . P^T, V^T read from the staged V
//           rows with ldmatrix.trans, the weights P split into bf16 high and
//           low parts the same way (two MMAs).
// Heads past G are zero rows of q and P. Once the scores are formed, the
// staging rows receive the tile's V rows (one asynchronous copy per tile)
// while the next tile's offsets are looked up and the softmax runs on the
// score fragments. Rows of tokens without K/V are zero-filled so the V sum
// sees finite values. Tokens are numbered list-major (token t of selected
// block i is i * ratio + t, blocks that are not complete masked out), then
// the tail.
template <int HD, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, 2)
    qsa_prefill_attn_tile_kernel(const float *__restrict__ q, const uint16_t *__restrict__ kc,
                                 const uint16_t *__restrict__ vc, const int32_t *__restrict__ table, int n_pages,
                                 int P, const int32_t *__restrict__ lists, float *__restrict__ out,
                                 uint32_t first_pos, uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq,
                                 uint32_t nkv, float inv_sqrt_d, int32_t *dev_status) {
  constexpr int NC = HD / 8;          // 16-byte chunks of a K or V row
  constexpr int ROWB = HD * 2 + 16;   // staged row stride in bytes
  constexpr int QROW = HD + 8;        // q row stride in bf16 elements (16 bytes of padding)
  constexpr int PROW = 40;            // weight row stride in bf16 elements: 32 tokens + 16 bytes
  constexpr int MT = HD / 16;         // 16-dimension tiles of the V sum
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char *kbuf = smem;
  __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(smem + static_cast<size_t>(kAttnWarps) * 32 * ROWB);
  __nv_bfloat16 *pb = qb + 2 * 8 * QROW;   // [warp][hi, lo][8 heads][PROW]
  long long *roff = reinterpret_cast<long long *>(pb + kAttnWarps * 2 * 8 * PROW);
  float *pm = reinterpret_cast<float *>(roff + 2 * kAttnWarps * 32);
  float *pl = pm + kAttnWarps * G;
  constexpr int PSTR = HD + 4;        // merge row stride in floats: the fragment stores hit distinct banks
  float *part = reinterpret_cast<float *>(smem);   // [warp][G][PSTR] after the tiles: aliases the staged rows
  static_assert(kAttnWarps * G * PSTR * 4 <= kAttnWarps * 32 * ROWB, "merge buffer fits the staging area");

  const int r = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long p = static_cast<long long>(first_pos) + r;
  for (int x = threadIdx.x; x < 8 * HD; x += kAttnWarps * 32) {
    const int g = x / HD, d = x % HD;
    const float v =
        g < G ? q[(static_cast<long long>(r) * nq + static_cast<long long>(kvh) * G + g) * HD + d] * inv_sqrt_d : 0.0f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    qb[g * QROW + d] = hi;
    qb[(8 + g) * QROW + d] = __float2bfloat16_rn(v - __bfloat162float(hi));   // v - hi is exact in f32
  }
  for (int x = threadIdx.x; x < kAttnWarps * 2 * 8 * PROW; x += kAttnWarps * 32)
    pb[x] = __float2bfloat16_rn(0.0f);   // rows of heads past G stay zero
  __syncthreads();

  const long long ncomp = (p + 1) / ratio;
  const long long n_list = static_cast<long long>(topk) * ratio;
  const long long tail0 = ncomp * ratio;
  const long long n_virt = n_list + (p + 1 - tail0);
  unsigned char *kw = kbuf + static_cast<size_t>(warp) * 32 * ROWB;
  __nv_bfloat16 *pw = pb + warp * 2 * 8 * PROW;
  long long *ow2 = roff + warp * 64;   // [2][32]: this tile's and the next tile's row offsets
  const uint32_t kaddr = static_cast<uint32_t>(__cvta_generic_to_shared(kw));
  const uint32_t qaddr = static_cast<uint32_t>(__cvta_generic_to_shared(qb));
  const uint32_t paddr = static_cast<uint32_t>(__cvta_generic_to_shared(pw));
  // MMA fragment coordinates: lane holds rows (lane >> 2) and (lane >> 2) + 8
  // of a 16-row tile and columns (heads) h0 = 2 * (lane & 3), h0 + 1.
  const int h0 = 2 * (lane & 3);
  // mo: the reference maxima of heads h0, h0 + 1; lo: this lane's share of
  // their sums; o: O^T fragments (dimension 16mt + row, head h0 + (i & 1)).
  float mo[2] = {-INFINITY, -INFINITY}, lo[2] = {0.0f, 0.0f}, o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[mt][i] = 0.0f;
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
  // (consecutive lanes: consecutive chunks of one row) as one asynchronous
  // group; rows without a token are zero-filled.
  auto stage = [&](const uint16_t *cache, const long long *offs) {
    for (int x = lane; x < 32 * NC; x += 32) {
      const int t = x / NC, c = x % NC;
      const long long src = offs[t];
      if (src >= 0)
        cp_async16(kw + t * ROWB + c * 16, cache + src + c * 8);
      else
        *reinterpret_cast<uint4 *>(kw + t * ROWB + c * 16) = make_uint4(0u, 0u, 0u, 0u);
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

    // ---- scores: S[32 tokens x 8 heads] ----
    // tokens 16mt + (lane >> 2) (+ 8 in [2..3]), heads h0 and h0 + 1; the
    // q high and low parts accumulate apart (four independent MMA chains)
    float c[2][4], cl[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[mt][i] = cl[mt][i] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      uint32_t bh[2], bl[2];   // q rows (heads) 0-7, dimensions 16ks .. 16ks + 15
      const uint32_t qa = qaddr + ((lane & 7) * QROW + ks * 16 + ((lane >> 3) & 1) * 8) * 2;
      ldsm_x2(bh, qa);
      ldsm_x2(bl, qa + 8 * QROW * 2);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t a[4];   // K rows 16mt .. 16mt + 15, dimensions 16ks .. 16ks + 15
        ldsm_x4(a, kaddr + (16 * mt + (lane & 15)) * ROWB + (ks * 2 + (lane >> 4)) * 16);
        mma_bf16(c[mt], a, bh);
        mma_bf16(cl[mt], a, bl);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[mt][i] += cl[mt][i];
    __syncwarp();   // every lane has read its K fragments: the V rows may land
    stage(vc, ow);
    const long long nbase = base + kAttnWarps * 32;
    const long long noff = nbase < n_virt ? token_offset(nbase) : -1;
    const uint32_t nlive = __ballot_sync(0xFFFFFFFFu, noff >= 0);
    ow2[32 * (buf ^ 1) + lane] = noff;

    // ---- softmax on the score fragments: a token without K/V scores -inf ----
    float sv[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 16 * mt + (lane >> 2) + 8 * (i >> 1);
        sv[mt][i] = ((live >> t) & 1u) ? c[mt][i] : -INFINITY;
      }
    float mx[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(fmaxf(sv[0][hh], sv[0][hh + 2]), fmaxf(sv[1][hh], sv[1][hh + 2]));
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xFFFFFFFFu, mx[hh], sh));
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (h0 + hh < G && mx[hh] > mo[hh] + kLazyMax) {   // the head's reference maximum moves up: rescale
        const float corr = expf(mo[hh] - mx[hh]);
        mo[hh] = mx[hh];
        lo[hh] *= corr;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][hh] *= corr;
          o[mt][hh + 2] *= corr;
        }
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hh = i & 1;
        if (h0 + hh >= G) continue;
        const int t = 16 * mt + (lane >> 2) + 8 * (i >> 1);
        const float x = sv[mt][i];
        const float e = x != -INFINITY ? expf(x - mo[hh]) : 0.0f;   // at most e^kLazyMax
        lo[hh] += e;
        const __nv_bfloat16 ehi = __float2bfloat16_rn(e);
        pw[(h0 + hh) * PROW + t] = ehi;
        pw[(8 + h0 + hh) * PROW + t] = __float2bfloat16_rn(e - __bfloat162float(ehi));
      }
    cp_async_wait_all();
    __syncwarp();   // the V rows and every lane's weights are in place

    // ---- V sum: O^T[hd x 8 heads] += V^T . P^T ----
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t bh[2], bl[2];   // P rows (heads) 0-7, tokens 16kk .. 16kk + 15
      const uint32_t pa = paddr + ((lane & 7) * PROW + kk * 16 + ((lane >> 3) & 1) * 8) * 2;
      ldsm_x2(bh, pa);
      ldsm_x2(bl, pa + 8 * PROW * 2);
      const int tok = 16 * kk + (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a[4];   // V^T: dimensions 16mt .. 16mt + 15, tokens 16kk .. 16kk + 15
        ldsm_x4_trans(a, kaddr + tok * ROWB + (16 * mt + ((lane >> 3) & 1) * 8) * 2);
        mma_bf16(o[mt], a, bh);
        mma_bf16(o[mt], a, bl);
      }
    }
    off = noff;   // the next tile rewrites the staging rows and weights after the __syncwarp at its top
    live = nlive;
  }

#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) lo[hh] += __shfl_xor_sync(0xFFFFFFFFu, lo[hh], sh);
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && dev_status) atomicOr(dev_status, IDX_STATUS_BAD_BLOCK);
  __syncthreads();   // every warp is done with its staged rows: part reuses them
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int g = h0 + (i & 1);
      if (g < G) part[(warp * G + g) * PSTR + 16 * mt + (lane >> 2) + 8 * (i >> 1)] = o[mt][i];
    }
  if (lane < 4) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      if (h0 + hh < G) {
        pm[warp * G + h0 + hh] = mo[hh];
        pl[warp * G + h0 + hh] = lo[hh];
      }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < G * HD; x += kAttnWarps * 32) {
    const int g = x / HD, d = x % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, pm[w * G + g]);
    float L = 0.0f, acc = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        if (pm[w * G + g] == -INFINITY) continue;   // a warp that saw no token
        const float cw = expf(pm[w * G + g] - M);
        L = fmaf(pl[w * G + g], cw, L);
        acc = fmaf(part[(w * G + g) * PSTR + d], cw, acc);
      }
    }
    out[(static_cast<long long>(r) * nq + static_cast<long long>(kvh) * G + g) * HD + d] = L > 0.0f ? acc / L : 0.0f;
  }
}

template <int HD, int G>
cudaError_t launch_tile(dim3 grid, cudaStream_t s, const float *q, const uint16_t *kc, const uint16_t *vc,
                        const int32_t *table, int n_pages, int P, const int32_t *lists, float *out,
                        uint32_t first_pos, uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq,
                        uint32_t nkv, float inv_sqrt_d, int32_t *dev_status) {
  constexpr size_t bytes = tile_smem_bytes<HD, G>();
  // set on every call: the attribute belongs to the current device's context
  const cudaError_t attr = cudaFuncSetAttribute(qsa_prefill_attn_tile_kernel<HD, G>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
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
  if (qsa_attn_tc_supported(q, nq, nkv, hd, k_cache, v_cache, rows, first_pos, topk, ratio, P, block_size)) {
    const cudaError_t e = launch_qsa_attn_tc(q, k_cache, v_cache, block_table, n_pages, P, lists, attn_out, rows,
                                             first_pos, topk, ratio, block_size, nq, nkv, inv_sqrt_d, dev_status, s);
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
  }
  if ((G == 1 || G == 2 || G == 4 || G == 8) && (hd == 64 || hd == 128) && aligned_to(k_cache, 16) &&
      aligned_to(v_cache, 16)) {   // both caches are staged by 16-byte asynchronous copies
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
