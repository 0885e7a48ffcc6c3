// topk.cu — TopK(I[t,:], k) from a score matrix, one thread-block cluster per
// query (or per piece of a very long query).
//
// Output order is the top-k write-out of "indexer_score_topk.cu": score
// descending, lower index first on equal scores, -1 / -inf padding. Both score
// paths write I[t, 0..valid_len) (with -inf for keys of out-of-range blocks)
// into a [T, ld] matrix; this file selects from it.
//
// A cluster of C CTAs (C <= 8) holds up to C * 4096 keys of one query in
// registers (16 per thread) and finds the k largest composite keys (see
// common.cuh) without re-reading them:
//   1. every CTA builds a 4096-bin shared-memory histogram of the next 12 key
//      bits of its keys;
//   2. every CTA adds its nonzero bins into the owners' sums (CTA r owns bins
//      [r*4096/C, (r+1)*4096/C)) with distributed shared-memory reductions,
//      and each owner publishes its slice total to all CTAs;
//   3. the CTA whose slice holds the k-th key locates that bin and publishes
//      it; if the bin holds more keys than the boundary buffer, the keys in it
//      are histogrammed again on the next 12 bits (still from registers);
//   4. when the first digit decides, every key at or above the boundary bin
//      goes straight into its bin's segment of a buffer in CTA 0, which ranks
//      each key inside its bin and writes it to its output slot; after a
//      refinement the keys are collected (one distributed shared-memory
//      atomic per warp) and CTA 0 sorts them (bitonic, short strides in
//      registers) and keeps the first k.
// A query longer than one cluster's reach is split into pieces whose k best
// keys go to a candidate list; the next launch selects from those lists the
// same way (each stage shrinks a query's keys at least 8-fold).
#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelR = 16;                           // keys per thread, in registers
constexpr int kCtaKeys = kSelThreads * kSelR;       // 4096
constexpr int kBins = 4096;                         // 12-bit digits
constexpr int kBndCap = 512;                        // largest boundary bin collected (else refine)
constexpr int kMaxCluster = 8;

// ------------------------------------------- cluster / DSMEM primitives ----
namespace cl {
__device__ __forceinline__ uint32_t rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster; orders shared-memory writes before
// the barrier (any CTA's) with reads after it.
__device__ __forceinline__ void sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
__device__ __forceinline__ void arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Address of the same shared-memory variable in CTA `r` of the cluster.
__device__ __forceinline__ uint32_t map(const void *p, uint32_t r) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(a)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(r));
  return a;
}
__device__ __forceinline__ void st_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_u64(uint32_t a, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ void red_add(uint32_t a, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add(uint32_t a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
  return old;
}
}  // namespace cl

__host__ __device__ inline int pow2_at_least(int k) {
  int kp = 1;
  while (kp < k) kp <<= 1;
  return kp;
}

struct SelShared {
  uint32_t hist[kBins];               // this CTA's histogram of the current digit
  uint32_t red[kBins / 2];            // cluster sums of this rank's slice of bins (C >= 2)
  uint32_t slice_tot[kMaxCluster];    // per rank: keys in its slice of bins
  uint32_t warp_sum[kSelThreads / 32];
  int b_bin, b_above, b_cnt;          // boundary bin, published by its owner
  int n_buf;                          // CTA 0: append cursor
};

// Dynamic shared memory: SelShared, then the collect buffer: up to k - 1
// keys above the boundary bin plus at most kBndCap keys in it, rounded up to a
// power of two (>= 64: the sort works on whole warps' 64-key segments).
struct SelSmem {
  size_t buf, total;
};
__host__ __device__ inline SelSmem sel_smem(int k) {
  SelSmem m{};
  m.buf = (sizeof(SelShared) + 15) & ~size_t(15);
  const int cap = k + kBndCap;
  m.total = m.buf + static_cast<size_t>(pow2_at_least(cap < 64 ? 64 : cap)) * 8;
  return m;
}

struct SelArgs {
  const float *scores;      // stage 0: [T, ld]
  long long ld;
  const uint64_t *cand_in;  // later stages: [T, n_in] keys (0 = none)
  long long n_in;
  uint64_t *cand_out;       // non-final stages: [T, gridDim.x / C, k] keys
};

__device__ __forceinline__ bool bad_len(const ScoreParams &p, int L) {
  return L < 0 || static_cast<long long>(L) > static_cast<long long>(p.max_lb) * p.epb;
}

// Sorts out[0 .. m) descending (m a power of two, 64 <= m): bitonic network,
// strides >= 64 through shared memory, strides <= 32 in registers (a warp
// holds 64 consecutive keys) so they need no block barrier.
__device__ void sort_desc(uint64_t *out, int m) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kSelThreads / 32;
  // in-register stages of one bitonic merge of `size`, strides 32 .. 1
  auto warp_phase = [&](int size, int smax) {
    for (int seg = warp; seg < (m >> 6); seg += kWarps) {
      const int e0 = seg * 64 + lane;          // elements e0 and e0 + 32
      uint64_t a = out[e0], b = out[e0 + 32];
      for (int sz = (size < 64 ? 2 : size); sz <= (size < 64 ? 64 : size); sz <<= 1) {
        for (int s = min(sz >> 1, smax); s > 0; s >>= 1) {
          if (s == 32) {
            const bool desc = ((e0 & sz) == 0);
            if ((a < b) == desc) {
              const uint64_t x = a;
              a = b;
              b = x;
            }
          } else {
            // partner lane ^ s; the lower element of the pair keeps the larger
            // key in a descending run
            const uint64_t pa = __shfl_xor_sync(0xFFFFFFFFu, a, s);
            const uint64_t pb = __shfl_xor_sync(0xFFFFFFFFu, b, s);
            const bool lower = (lane & s) == 0;
            const bool da = ((e0 & sz) == 0), db = (((e0 + 32) & sz) == 0);
            a = (lower == da) ? (a > pa ? a : pa) : (a < pa ? a : pa);
            b = (lower == db) ? (b > pb ? b : pb) : (b < pb ? b : pb);
          }
        }
      }
      out[e0] = a;
      out[e0 + 32] = b;
    }
  };
  warp_phase(0, 32);   // sizes 2 .. 64 entirely in registers
  __syncthreads();
  for (int size = 128; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride >= 64; stride >>= 1) {
      for (int i = tid; i < (m >> 1); i += kSelThreads) {
        const int lo = ((i & ~(stride - 1)) << 1) | (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = out[lo], b = out[hi];
        if ((a < b) == desc) {
          out[lo] = b;
          out[hi] = a;
        }
      }
      __syncthreads();
    }
    warp_phase(size, 32);
    __syncthreads();
  }
}

template <int C, bool kFromCand, bool kFinal>
__global__ void __launch_bounds__(kSelThreads, C == 1 ? 2 : (C == 2 ? 3 : 4)) topk_cluster_kernel(ScoreParams p, SelArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelShared *sh = reinterpret_cast<SelShared *>(smem_raw);
  const SelSmem lay = sel_smem(p.top_k);
  uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw + lay.buf);
  const uint32_t r = cl::rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.y;
  const int piece = blockIdx.x / C;
  const int k = p.top_k;
  // This kernel may be launched before the one writing its input has ended:
  // wait for that kernel's completion and memory first.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- this CTA's keys ----
  // Row positions are loaded up to the row capacity (max_lb * epb <= ld) and
  // masked by the valid length afterwards, so the loads need not wait for it.
  const long long lo = static_cast<long long>(piece) * C * kCtaKeys + static_cast<long long>(r) * kCtaKeys;
  const long long cap = kFromCand ? a.n_in : static_cast<long long>(p.max_lb) * p.epb;
  const long long hi_cap = min(cap, lo + kCtaKeys);
  float sv[kFromCand ? 1 : kSelR];
  uint64_t key[kSelR];
#pragma unroll
  for (int j = 0; j < kSelR; ++j) {
    const long long i = lo + j * kSelThreads + tid;
    if (kFromCand) {
      key[j] = (i < hi_cap) ? a.cand_in[static_cast<long long>(t) * a.n_in + i] : 0ull;
    } else {
      sv[kFromCand ? 0 : j] = (i < hi_cap) ? a.scores[static_cast<long long>(t) * a.ld + i] : -INFINITY;
    }
  }
  if (!kFromCand) {
    const int L = p.valid_lens[t];
    if (bad_len(p, L)) {  // uniform over the cluster: nobody reaches a cluster barrier
      if (r == 0) {
        if (kFinal) {
          if (tid == 0 && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_LEN);
          for (int i = tid; i < k; i += kSelThreads) {
            p.topk_idx[static_cast<long long>(t) * k + i] = -1;
            p.topk_score[static_cast<long long>(t) * k + i] = -INFINITY;
          }
        } else {
          if (piece == 0 && tid == 0 && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_LEN);
          uint64_t *dst = a.cand_out + (static_cast<long long>(t) * (gridDim.x / C) + piece) * k;
          for (int i = tid; i < k; i += kSelThreads) dst[i] = 0ull;
        }
      }
      return;
    }
#pragma unroll
    for (int j = 0; j < kSelR; ++j) {
      const long long i = lo + j * kSelThreads + tid;
      const float v = sv[kFromCand ? 0 : j];
      key[j] = (i < L && v != -INFINITY) ? pack_key(v, static_cast<int32_t>(i)) : 0ull;
    }
  }
  if (r == 0 && tid == 0) sh->n_buf = 0;

  // ---- locate the boundary bin, digit by digit ----
  constexpr int sl = kBins / C;             // bins per rank
  constexpr int per = sl / kSelThreads;     // bins per thread (>= 2)
  const int bin_top = (static_cast<int>(r) + 1) * sl - 1;
  uint64_t prefix = 0, mask = 0;
  int need = k, shift = 52, width = 12, rounds = 0;
  uint32_t all_keys = 0;
  bool take_all = false;
  if (C > 1)
    for (int b = tid; b < sl; b += kSelThreads) sh->red[b] = 0u;
  cl::arrive();  // every CTA's sums are zero (and it has started) before anyone adds into them
  bool first = true;
  while (true) {
    for (int b = tid; b < kBins; b += kSelThreads) sh->hist[b] = 0u;
    __syncthreads();
    const uint32_t dmask = (1u << width) - 1u;
#pragma unroll
    for (int j = 0; j < kSelR; ++j)
      if (key[j] != 0ull && (key[j] & mask) == prefix)
        atomicAdd(&sh->hist[static_cast<uint32_t>(key[j] >> shift) & dmask], 1u);
    __syncthreads();
    if (first) {
      cl::wait();
      first = false;
    }
    if (C > 1) {  // add every nonzero bin into its owner's sums (no round trip)
#pragma unroll
      for (int j = 0; j < kBins / kSelThreads; ++j) {
        const int b = tid + j * kSelThreads;
        const uint32_t v = sh->hist[b];
        if (v != 0u) cl::red_add(cl::map(&sh->red[b % sl], static_cast<uint32_t>(b / sl)), v);
      }
    }
    cl::sync();
    // my slice's cluster sums; thread tid owns bins bin_top - per*tid - j
    uint32_t c[per];
    uint32_t tot = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      const int lb = sl - 1 - per * tid - j;   // index within the slice
      if (C > 1) {
        c[j] = sh->red[lb];
        sh->red[lb] = 0u;                       // ready for the next digit's sums
      } else {
        c[j] = sh->hist[lb];
      }
      tot += c[j];
    }
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sh->warp_sum[warp] = incl;
    __syncthreads();
    uint32_t before = 0, slice = 0;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) {
      const uint32_t s = sh->warp_sum[w];
      if (w < warp) before += s;
      slice += s;
    }
    if (tid < C) cl::st_u32(cl::map(&sh->slice_tot[r], tid), slice);
    cl::sync();
    uint32_t above = 0, all = 0;
#pragma unroll
    for (int q = 0; q < C; ++q) {
      const uint32_t s = sh->slice_tot[q];
      if (q > static_cast<int>(r)) above += s;
      all += s;
    }
    uint32_t run = above + before + incl - tot;
    if (shift == 52) {
      // First digit: publish, for every bin that holds some of the k best
      // keys, its place in the output (keys in higher bins) and its count,
      // packed as start | count << 16, into CTA 0's histogram array (no CTA
      // reads histograms any more this round).
      uint32_t rb = run;
#pragma unroll
      for (int j = 0; j < per; ++j) {
        if (c[j] != 0u && rb < static_cast<uint32_t>(k))
          cl::st_u32(cl::map(&sh->hist[bin_top - per * tid - j], 0), rb | (c[j] << 16));
        rb += c[j];
      }
    }
    all_keys = all;
    if (all <= static_cast<uint32_t>(need)) {
      take_all = true;  // every key matching the prefix is selected (same decision in every CTA)
      cl::sync();
      break;
    }
#pragma unroll
    for (int j = 0; j < per; ++j) {
      if (run < static_cast<uint32_t>(need) && run + c[j] >= static_cast<uint32_t>(need)) {
        const int b = bin_top - per * tid - j;
        for (int q = 0; q < C; ++q) {
          cl::st_u32(cl::map(&sh->b_bin, q), static_cast<uint32_t>(b));
          cl::st_u32(cl::map(&sh->b_above, q), run);
          cl::st_u32(cl::map(&sh->b_cnt, q), c[j]);
        }
      }
      run += c[j];
    }
    cl::sync();
    const int bin = sh->b_bin, cnt = sh->b_cnt;
    prefix |= static_cast<uint64_t>(bin) << shift;
    mask |= static_cast<uint64_t>(dmask) << shift;
    ++rounds;
    if (cnt <= kBndCap || shift == 0) break;
    need -= sh->b_above;
    // digits: bits 63..52, 51..40, 39..28, 27..16, 15..4, then 3..0
    if (shift >= 12) {
      shift -= 12;
      width = 12;
    } else {
      width = shift;
      shift = 0;
    }
    // the histogram is cleared next round: every CTA has finished reading it
    // (the reads precede the barrier just passed)
  }

  // ---- decided on the first digit, with a small boundary bin: rank path ----
  // Every key at or above the boundary bin goes straight into its bin's
  // segment of CTA 0's buffer (bins in descending order); CTA 0 then ranks
  // each key inside its bin and writes it to its final place. No sort.
  if ((take_all && rounds == 0) || (!take_all && rounds == 1)) {
    const uint32_t table = cl::map(sh->hist, 0), buf_r = cl::map(buf, 0);
#pragma unroll
    for (int j = 0; j < kSelR; ++j) {
      if (key[j] != 0ull && (key[j] & mask) >= prefix) {
        const uint32_t old = cl::atom_add(table + 4u * static_cast<uint32_t>(key[j] >> 52), 1u);
        cl::st_u64(buf_r + 8u * (old & 0xFFFFu), key[j]);
      }
    }
    cl::sync();
    if (r != 0) return;
    const int total = take_all ? static_cast<int>(all_keys) : sh->b_above + sh->b_cnt;
    uint64_t *dst = kFinal ? nullptr : a.cand_out + (static_cast<long long>(t) * (gridDim.x / C) + piece) * k;
    for (int p0 = tid; p0 < total; p0 += kSelThreads) {
      const uint64_t kv = buf[p0];
      const uint32_t pk = sh->hist[kv >> 52];
      const int end = static_cast<int>(pk & 0xFFFFu), start = end - static_cast<int>(pk >> 16);
      int pos = start, q = start;
      for (; q + 8 <= end; q += 8) {   // eight loads in flight per step
        uint64_t x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = buf[q + u];
#pragma unroll
        for (int u = 0; u < 8; ++u) pos += (x[u] > kv) ? 1 : 0;
      }
      for (; q < end; ++q) pos += (buf[q] > kv) ? 1 : 0;
      if (pos < k) {
        if (kFinal) {
          p.topk_idx[static_cast<long long>(t) * k + pos] = key_index(kv);
          p.topk_score[static_cast<long long>(t) * k + pos] = key_score(kv);
        } else {
          dst[pos] = kv;
        }
      }
    }
    for (int i = total + tid; i < k; i += kSelThreads) {
      if (kFinal) {
        p.topk_idx[static_cast<long long>(t) * k + i] = -1;
        p.topk_score[static_cast<long long>(t) * k + i] = -INFINITY;
      } else {
        dst[i] = 0ull;
      }
    }
    return;
  }

  // ---- otherwise collect into CTA 0 every key at or above the boundary bin ----
  // (one cluster atomic per warp: count first, then place)
  const uint32_t buf_base = cl::map(buf, 0), nbuf_a = cl::map(&sh->n_buf, 0);
  uint32_t total = 0;
#pragma unroll
  for (int j = 0; j < kSelR; ++j)
    total += __popc(__ballot_sync(0xFFFFFFFFu, key[j] != 0ull && (key[j] & mask) >= prefix));
  uint32_t base = 0;
  if (lane == 0 && total) base = cl::atom_add(nbuf_a, total);
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  const uint32_t below = lanemask_lt();
#pragma unroll
  for (int j = 0; j < kSelR; ++j) {
    const bool take = key[j] != 0ull && (key[j] & mask) >= prefix;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
    if (take) cl::st_u64(buf_base + 8u * (base + __popc(m & below)), key[j]);
    base += __popc(m);
  }
  cl::sync();
  if (r != 0) return;  // nothing touches this CTA's shared memory any more

  // ---- CTA 0: sort what was collected (all keys above the boundary bin and
  // every key in it) and keep the first k ----
  const int count = sh->n_buf;
  const int m = max(64, pow2_at_least(count));
  for (int i = count + tid; i < m; i += kSelThreads) buf[i] = 0ull;
  __syncthreads();
  sort_desc(buf, m);
  const int kept = min(count, k);
  if (kFinal) {
    int32_t *oi = p.topk_idx + static_cast<long long>(t) * k;
    float *os = p.topk_score + static_cast<long long>(t) * k;
    for (int i = tid; i < k; i += kSelThreads) {
      if (i < kept) {
        const uint64_t kv = buf[i];
        oi[i] = key_index(kv);
        os[i] = key_score(kv);
      } else {
        oi[i] = -1;
        os[i] = -INFINITY;
      }
    }
  } else {
    uint64_t *dst = a.cand_out + (static_cast<long long>(t) * (gridDim.x / C) + piece) * k;
    for (int i = tid; i < k; i += kSelThreads) dst[i] = (i < kept) ? buf[i] : 0ull;
  }
}

template <int C, bool kFromCand, bool kFinal>
cudaError_t launch_stage_c(const ScoreParams &p, const SelArgs &a, int pieces, size_t smem, cudaStream_t stream) {
  auto fn = topk_cluster_kernel<C, kFromCand, kFinal>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(C * pieces), static_cast<unsigned>(p.T), 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the previous kernel's tail
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, p, a);
}

template <bool kFromCand, bool kFinal>
cudaError_t launch_stage(const ScoreParams &p, const SelArgs &a, int C, int pieces, size_t smem,
                         cudaStream_t stream) {
  switch (C) {
    case 1: return launch_stage_c<1, kFromCand, kFinal>(p, a, pieces, smem, stream);
    case 2: return launch_stage_c<2, kFromCand, kFinal>(p, a, pieces, smem, stream);
    case 4: return launch_stage_c<4, kFromCand, kFinal>(p, a, pieces, smem, stream);
    case 8: return launch_stage_c<8, kFromCand, kFinal>(p, a, pieces, smem, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

// Stage shape for n keys per query: cluster size and number of pieces.
// The cluster size is a power of two so that it divides the 4096 bins.
void stage_shape(long long n, int *C, long long *pieces) {
  long long c = 1;
  while (c < kMaxCluster && c * kCtaKeys < n) c <<= 1;
  *C = static_cast<int>(c);
  long long pc = (n + c * kCtaKeys - 1) / (c * kCtaKeys);
  *pieces = pc < 1 ? 1 : pc;
}

}  // namespace

SelectPlan select_plan(int T, int top_k, long long max_len, bool have_scores_out, long long ld_out) {
  SelectPlan pl{};
  pl.own_scores = !have_scores_out;
  pl.ld = have_scores_out ? ld_out : max_len;
  long long n = max_len;
  long long biggest[2] = {0, 0};  // largest candidate list sizes (keys per query) of even / odd stages
  pl.n_stages = 0;
  while (pl.n_stages < kMaxSelectStages) {
    int C;
    long long pieces;
    stage_shape(n, &C, &pieces);
    pl.C[pl.n_stages] = C;
    pl.pieces[pl.n_stages] = static_cast<int>(pieces);
    pl.n_in[pl.n_stages] = n;
    ++pl.n_stages;
    if (pieces == 1) break;
    n = pieces * top_k;
    long long &b = biggest[(pl.n_stages - 1) & 1];
    if (n > b) b = n;
  }
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  pl.scores_off = off;
  if (pl.own_scores) off = al(off + static_cast<size_t>(T) * static_cast<size_t>(max_len) * 4);
  for (int i = 0; i < 2; ++i) {
    pl.cand_off[i] = off;
    off = al(off + static_cast<size_t>(T) * static_cast<size_t>(biggest[i]) * 8);
  }
  pl.total = off;
  return pl;
}

bool select_supported(int top_k, long long max_len) {
  SelectPlan pl = select_plan(1, top_k, max_len, true, max_len);
  int C;
  long long pieces;
  stage_shape(pl.n_in[pl.n_stages - 1], &C, &pieces);
  return pieces == 1 && sel_smem(top_k).total <= 227 * 1024;
}

cudaError_t launch_select(const ScoreParams &p, const float *scores, long long ld, const SelectPlan &pl,
                          void *workspace, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  const size_t smem = sel_smem(p.top_k).total;
  unsigned char *base = static_cast<unsigned char *>(workspace);
  cudaError_t e = cudaSuccess;
  for (int s = 0; s < pl.n_stages && e == cudaSuccess; ++s) {
    SelArgs a{};
    a.scores = scores;
    a.ld = ld;
    a.n_in = pl.n_in[s];
    if (s > 0) a.cand_in = reinterpret_cast<const uint64_t *>(base + pl.cand_off[(s - 1) & 1]);
    const bool final = (s == pl.n_stages - 1);
    if (!final) a.cand_out = reinterpret_cast<uint64_t *>(base + pl.cand_off[s & 1]);
    if (s == 0 && final) e = launch_stage<false, true>(p, a, pl.C[s], pl.pieces[s], smem, stream);
    else if (s == 0) e = launch_stage<false, false>(p, a, pl.C[s], pl.pieces[s], smem, stream);
    else if (final) e = launch_stage<true, true>(p, a, pl.C[s], pl.pieces[s], smem, stream);
    else e = launch_stage<true, false>(p, a, pl.C[s], pl.pieces[s], smem, stream);
  }
  return e;
}

}  // namespace idx
