// topk.cu — TopK(I[t,:], k) from a score matrix: one CTA per query streams
// its row.
//
// Output order is the top-k write-out of "indexer_score_topk.cu": score
// descending, lower index first on equal scores, -1 / -inf padding. Both score
// paths write I[t, 0..valid_len) (with -inf for keys of out-of-range blocks)
// into a [T, ld] matrix; this file selects from it.
//
// The k largest composite keys (see common.cuh) are found digit by digit,
// 12 key bits at a time, without holding the row:
//   1. the histogram of the first digit comes from the tensor-core scorer
//      (which counts every key it writes), or from one pass over the row;
//      a descending scan over the 4096 bins locates the bin holding the k-th
//      key (the boundary bin) and the place in the output of every bin above;
//   2. if the boundary bin holds more than kBndCap keys, its keys are
//      histogrammed on the next digit (another pass) until it does not;
//   3. decided on the first digit (the usual case): one pass drops every key
//      at or above the boundary bin straight into its bin's segment of a
//      shared-memory buffer (bins in descending order); each key is then
//      ranked inside its bin — the boundary bin first split by the next 8
//      bits — and written to its output slot. No sort.
//      Decided on a later digit: one pass collects the keys at or above the
//      boundary and a bitonic sort orders them.
#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kThreads = 512;
constexpr int kBins = kScoreBins;                 // 12-bit digits
constexpr int kPer = kBins / kThreads;            // bins each thread owns in a scan
constexpr int kBndCap = 512;                      // largest boundary bin collected (else refine)
constexpr int kUnroll = 8;                        // score loads in flight per thread
static_assert(kBndCap <= kThreads, "the boundary-bin split holds one key per thread");

__host__ __device__ inline int pow2_at_least(int k) {
  int kp = 1;
  while (kp < k) kp <<= 1;
  return kp;
}

struct SelShared {
  uint32_t table[kBins];      // counts of the current digit; once the first digit decides,
                              // per bin: end of its buffer segment | count << 16
  uint32_t warp_sum[kThreads / 32];
  uint32_t sub_cnt[256], sub_cur[256];  // the boundary bin's split by the next 8 bits
  int b_bin, b_above, b_cnt;  // boundary bin, its keys above, its keys
  int n_buf;                  // append cursor (later-digit decisions)
};

// Dynamic shared memory: SelShared, then the key buffer: up to k - 1 keys
// above the boundary bin plus at most kBndCap keys in it, rounded up to a
// power of two (>= 64: the sort works on whole warps' 64-key segments).
struct SelSmem {
  size_t buf, cap, total;  // cap: keys the buffer holds
};
__host__ __device__ inline SelSmem sel_smem(int k) {
  SelSmem m{};
  m.buf = (sizeof(SelShared) + 15) & ~size_t(15);
  const int want = k + kBndCap;
  m.cap = static_cast<size_t>(pow2_at_least(want < 64 ? 64 : want));
  m.total = m.buf + m.cap * 8;
  return m;
}

// Sorts out[0 .. m) descending (m a power of two, 64 <= m): bitonic network,
// strides >= 64 through shared memory, strides <= 32 in registers (a warp
// holds 64 consecutive keys) so they need no block barrier.
__device__ void sort_desc(uint64_t *out, int m) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kThreads / 32;
  // in-register stages of the bitonic merges: sizes 2 .. 64 when size < 64,
  // else the strides 32 .. 1 of one merge of `size`
  auto warp_phase = [&](int size) {
    for (int seg = warp; seg < (m >> 6); seg += kWarps) {
      const int e0 = seg * 64 + lane;  // elements e0 and e0 + 32
      uint64_t a = out[e0], b = out[e0 + 32];
      for (int sz = (size < 64 ? 2 : size); sz <= (size < 64 ? 64 : size); sz <<= 1) {
        for (int s = min(sz >> 1, 32); s > 0; s >>= 1) {
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
  warp_phase(0);
  __syncthreads();
  for (int size = 128; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride >= 64; stride >>= 1) {
      for (int i = tid; i < (m >> 1); i += kThreads) {
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
    warp_phase(size);
    __syncthreads();
  }
}

__device__ __forceinline__ bool bad_len(const ScoreParams &p, int L) {
  return L < 0 || static_cast<long long>(L) > static_cast<long long>(p.max_lb) * p.epb;
}

// Calls f(key) for every key of row[0 .. L) that is not -inf, kUnroll loads
// in flight per thread.
template <class F>
__device__ __forceinline__ void for_each_key(const float *row, int L, F &&f) {
  for (long long base = 0; base < L; base += kThreads * kUnroll) {
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = base + u * kThreads + threadIdx.x;
      v[u] = (i < L) ? row[i] : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = base + u * kThreads + threadIdx.x;
      if (v[u] != -INFINITY) f(pack_key(v[u], static_cast<int32_t>(i)));
    }
  }
}


__global__ void __launch_bounds__(kThreads) topk_stream_kernel(ScoreParams p, const float *__restrict__ scores,
                                                              long long ld, const uint32_t *__restrict__ hist) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelShared *sh = reinterpret_cast<SelShared *>(smem_raw);
  const SelSmem lay = sel_smem(p.top_k);
  uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw + lay.buf);
  const int cap = static_cast<int>(lay.cap);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x;
  const int k = p.top_k;
  int32_t *oi = p.topk_idx + static_cast<long long>(t) * k;
  float *os = p.topk_score + static_cast<long long>(t) * k;
  // This kernel may be launched before the one writing its input has ended:
  // wait for that kernel's completion and memory first.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int L = p.valid_lens[t];
  if (bad_len(p, L)) {
    if (tid == 0 && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_LEN);
    for (int i = tid; i < k; i += kThreads) {
      oi[i] = -1;
      os[i] = -INFINITY;
    }
    return;
  }
  const float *row = scores + static_cast<long long>(t) * ld;
  if (tid == 0) {
    sh->b_bin = 0;
    sh->b_above = 0;
    sh->b_cnt = 0;
    sh->n_buf = 0;
  }

  // ---- locate the boundary bin, digit by digit ----
  // In a scan thread tid owns bins kBins-1-kPer*tid-j (j < kPer): descending.
  uint64_t prefix = 0, mask = 0;
  int need = k, shift = 52, width = 12, rounds = 0;
  uint32_t all_keys = 0;
  bool take_all = false;
  while (true) {
    const uint32_t dmask = (1u << width) - 1u;
    uint32_t c[kPer];
    if (rounds == 0 && hist != nullptr) {
      const uint32_t *h = hist + static_cast<size_t>(t) * kBins;
#pragma unroll
      for (int j = 0; j < kPer; ++j) c[j] = h[kBins - 1 - kPer * tid - j];
    } else {
      for (int b = tid; b < kBins; b += kThreads) sh->table[b] = 0u;
      __syncthreads();
      for_each_key(row, L, [&](uint64_t key) {
        if ((key & mask) == prefix) atomicAdd(&sh->table[static_cast<uint32_t>(key >> shift) & dmask], 1u);
      });
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kPer; ++j) c[j] = sh->table[kBins - 1 - kPer * tid - j];
    }
    uint32_t tot = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) tot += c[j];
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sh->warp_sum[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      const uint32_t s = sh->warp_sum[w];
      if (w < warp) before += s;
      all += s;
    }
    const uint32_t run0 = before + incl - tot;   // keys in higher bins
    if (rounds == 0) {
      // First digit: for every bin holding some of the k best keys, the end
      // of its segment (before any key is placed: its start) | its count.
      // Each thread rewrites only the bins it owns and has already read.
      uint32_t rb = run0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (c[j] != 0u && rb < static_cast<uint32_t>(k)) sh->table[kBins - 1 - kPer * tid - j] = rb | (c[j] << 16);
        rb += c[j];
      }
    }
    all_keys = all;
    if (all <= static_cast<uint32_t>(need)) {
      take_all = true;  // every key matching the prefix is selected
      __syncthreads();
      break;
    }
    uint32_t run = run0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (run < static_cast<uint32_t>(need) && run + c[j] >= static_cast<uint32_t>(need)) {
        sh->b_bin = kBins - 1 - kPer * tid - j;
        sh->b_above = static_cast<int>(run);
        sh->b_cnt = static_cast<int>(c[j]);
      }
      run += c[j];
    }
    __syncthreads();
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
    __syncthreads();   // every thread has read this round's boundary before the table is reused
  }

  auto emit = [&](uint64_t kv, int pos) {
    if (pos < k) {
      oi[pos] = key_index(kv);
      os[pos] = key_score(kv);
    }
  };
  int produced;  // output slots filled; the rest is padding

  if ((take_all && rounds == 0) || (!take_all && rounds == 1)) {
    // ---- decided on the first digit: place, rank, write ----
    for_each_key(row, L, [&](uint64_t key) {
      if ((key & mask) >= prefix) {
        const uint32_t old = atomicAdd(&sh->table[key >> 52], 1u);
        if (static_cast<int>(old & 0xFFFFu) < cap) buf[old & 0xFFFFu] = key;
      }
    });
    __syncthreads();
    const int total = min(take_all ? static_cast<int>(all_keys) : sh->b_above + sh->b_cnt, cap);
    // rank of kv among buf[q0 .. q1): keys above it
    auto rank_in = [&](uint64_t kv, int q0, int q1) {
      int n = 0, q = q0;
      for (; q + 8 <= q1; q += 8) {  // eight loads in flight per step
        uint64_t x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = buf[q + u];
#pragma unroll
        for (int u = 0; u < 8; ++u) n += (x[u] > kv) ? 1 : 0;
      }
      for (; q < q1; ++q) n += (buf[q] > kv) ? 1 : 0;
      return n;
    };
    // The boundary bin (often a few hundred keys) is first ordered by the
    // next 8 key bits, so each of its keys is ranked only among keys sharing
    // those too.
    const int bs = take_all ? total : min(sh->b_above, total), be = total;
    const bool split = be - bs > 64;
    if (split) {
      if (tid < 256) sh->sub_cnt[tid] = 0u;
      __syncthreads();
      const bool mine = bs + tid < be;       // one boundary key per thread
      const uint64_t bk = mine ? buf[bs + tid] : 0ull;
      const uint32_t sd = static_cast<uint32_t>(bk >> 44) & 255u;
      if (mine) atomicAdd(&sh->sub_cnt[sd], 1u);
      __syncthreads();
      if (warp == 0) {  // descending exclusive scan: sub-bin d starts after all keys of sub-bins > d
        uint32_t c8[8], tot = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          c8[u] = sh->sub_cnt[255 - 8 * lane - u];
          tot += c8[u];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += v;
        }
        uint32_t r = incl - tot;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sh->sub_cur[255 - 8 * lane - u] = r;
          r += c8[u];
        }
      }
      __syncthreads();
      const uint32_t spos = mine ? atomicAdd(&sh->sub_cur[sd], 1u) : 0u;
      __syncthreads();  // every boundary key is in a register: its segment may be rewritten
      if (mine) buf[bs + static_cast<int>(spos)] = bk;
      __syncthreads();
      if (mine) {  // sub_cur[sd] now ends sub-bin sd's run; it starts sub_cnt[sd] earlier
        const int q1 = bs + static_cast<int>(sh->sub_cur[sd]), q0 = q1 - static_cast<int>(sh->sub_cnt[sd]);
        emit(bk, q0 + rank_in(bk, q0, q1));
      }
    }
    for (int p0 = tid; p0 < (split ? bs : total); p0 += kThreads) {
      const uint64_t kv = buf[p0];
      const uint32_t pk = sh->table[kv >> 52];
      const int end = min(static_cast<int>(pk & 0xFFFFu), total);
      const int start = max(0, static_cast<int>(pk & 0xFFFFu) - static_cast<int>(pk >> 16));
      emit(kv, start + rank_in(kv, start, end));
    }
    produced = min(total, k);
  } else {
    // ---- decided on a later digit: collect, sort, write ----
    for_each_key(row, L, [&](uint64_t key) {
      if ((key & mask) >= prefix) {
        const int slot = atomicAdd(&sh->n_buf, 1);
        if (slot < cap) buf[slot] = key;
      }
    });
    __syncthreads();
    const int count = min(sh->n_buf, cap);
    const int m = max(64, pow2_at_least(count));
    for (int i = count + tid; i < m; i += kThreads) buf[i] = 0ull;
    __syncthreads();
    sort_desc(buf, m);
    produced = min(count, k);
    for (int i = tid; i < produced; i += kThreads) emit(buf[i], i);
  }
  for (int i = produced + tid; i < k; i += kThreads) {
    oi[i] = -1;
    os[i] = -INFINITY;
  }
}

}  // namespace

SelectPlan select_plan(int T, int top_k, long long max_len, bool have_scores_out, long long ld_out) {
  (void)top_k;
  SelectPlan pl{};
  pl.own_scores = !have_scores_out;
  pl.ld = have_scores_out ? ld_out : max_len;
  pl.scores_off = 0;
  pl.total = pl.own_scores ? ((static_cast<size_t>(T) * static_cast<size_t>(max_len) * 4 + 255) & ~size_t(255)) : 0;
  return pl;
}

bool select_supported(int top_k, long long max_len) {
  (void)max_len;
  return sel_smem(top_k).total <= 227 * 1024;
}

cudaError_t launch_select(const ScoreParams &p, const float *scores, long long ld, const uint32_t *hist,
                          const SelectPlan &pl, void *workspace, cudaStream_t stream) {
  (void)pl;
  (void)workspace;
  if (p.T == 0) return cudaSuccess;
  const size_t smem = sel_smem(p.top_k).total;
  cudaError_t e =
      cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.T), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the scorer's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_stream_kernel, p, scores, ld, hist);
}

}  // namespace idx
