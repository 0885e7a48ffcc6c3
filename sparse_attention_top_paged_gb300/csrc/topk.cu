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
//   3. decided on the first digit with no bin above the boundary holding more
//      than kRankBinMax keys (the decode case): one pass drops every key at
//      or above the boundary bin straight into its bin's segment of a
//      shared-memory buffer (bins in descending order); bins of more than
//      kWarpBin keys are first split on the next 8 key bits by the whole CTA
//      (more than kMaxLarge such bins: one bitonic sort of the buffer); then
//      each warp sorts whole bins in registers, one at a time, and writes
//      every key to its output slot (its bin's start + its rank in the bin).
//      Otherwise: one pass collects the keys at or above the boundary and a
//      bitonic sort orders them.
//      When rows leave SMs idle, several CTAs take each row (2 when each has
//      to stream the row, up to 4 when they read a list collected beforehand):
//      all decide the boundary alike, then CTA h places, orders and writes the
//      bins whose segment starts in part h of the buffer.
// Rows of at most kSmallRow keys skip the digits: every candidate key goes
// into the buffer and one bitonic sort orders them.
// Each pass reads the row from shared memory: one bulk copy stages the whole
// row when it holds at most kStageMax scores (else the row goes through in
// chunks of that size, one copy each), and the first copy is issued before
// the first digit is decided. For a few very long rows, select_collect_kernel
// (below) gathers step 3's keys beforehand over many CTAs, and the pass over
// the row becomes a pass over that list.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace idx {
namespace {

constexpr int kMaxThreads = 1024;                // selection CTA: 1024 threads when every row has an SM, else 512
constexpr int kBins = kScoreBins;                 // 12-bit digits
constexpr int kBndCap = 2048;                     // largest boundary bin collected (else refine)
constexpr int kRankBinMax = kBndCap;              // largest bin above the boundary ordered in place
constexpr int kMaxLarge = 8;                      // more larger bins than this: sort the whole buffer
constexpr int kMaxParts = 4;                      // CTAs that share one row's ordering (8 measured slower on long decode)
constexpr int kUnroll = 4;                        // 16-byte score loads in flight per thread
constexpr int kSmallRow = 2048;                   // rows up to this long are sorted whole
constexpr int kCollectThreads = 256;              // split collection: threads per CTA,
constexpr int kCollectMin = 2048;                 // at least this many keys per CTA,
constexpr int kMaxChunks = 32;                    // at most this many CTAs per row
constexpr int kCollectBuf = 2048;                 // keys a collecting CTA holds before flushing
constexpr long long kSplitMinLen = 65536;         // split only rows at least this long

__host__ __device__ inline int pow2_at_least(int k) {
  int kp = 1;
  while (kp < k) kp <<= 1;
  return kp;
}

struct SelShared {
  uint32_t table[kBins];      // counts of the current digit; once the first digit decides,
                              // per bin: end of its buffer segment | count << 16
  uint32_t warp_sum[kMaxThreads / 32];
  uint32_t warp_max[kMaxThreads / 32];   // largest bin above the boundary (first digit)
  int b_bin, b_above, b_cnt;  // boundary bin, its keys above, its keys
  int n_buf;                  // append cursor (later-digit decisions)
  int abort_flag;             // a staging copy never completed
  uint32_t sub_cnt[256], sub_cur[256];  // a large bin's split by the next 8 key bits
  int n_large;
  uint32_t large[8];          // packed entries of the large bins (kMaxLarge)
  int split_bin[kMaxParts];   // several CTAs a row: split_bin[q], the highest bin of part q (q >= 1)
};

// Dynamic shared memory: SelShared, then the key buffer: up to k - 1 keys
// above the boundary bin plus at most kBndCap keys in it, rounded up to a
// power of two (>= 64: the sort works on whole warps' 64-key segments).
// Then the row staging area (a whole row of up to kStageMax scores, else
// chunks of that size, copied in by one bulk copy each) and its mbarrier.
constexpr int kStageMax = 32768;
struct SelSmem {
  size_t buf, cap, stage, stage_floats, bar, total;  // cap: keys the buffer holds
};
__host__ __device__ inline SelSmem sel_smem(int k, long long max_len) {
  SelSmem m{};
  m.buf = (sizeof(SelShared) + 127) & ~size_t(127);   // 128-byte aligned: a warp's 16-byte reads of the staged row then span whole lines
  const int want = k + kBndCap;
  m.cap = static_cast<size_t>(pow2_at_least(want < 64 ? 64 : want));
  m.stage = m.buf + m.cap * 8;
  const long long sf = (max_len + 3) & ~3LL;
  m.stage_floats = static_cast<size_t>(sf < kStageMax ? sf : kStageMax);
  m.bar = m.stage + m.stage_floats * 4;
  m.total = m.bar + 8;
  return m;
}

// Sorts out[0 .. m) descending (m a power of two, 64 <= m): bitonic network,
// strides >= 64 through shared memory, strides <= 32 in registers (a warp
// holds 64 consecutive keys) so they need no block barrier.
template <int kThreads>
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

// The scores of one row, read pass by pass. A 16-byte-aligned row comes in
// through bulk copies into shared memory, kStageMax scores at a time (a row
// that fits stays resident across passes; the first copy is issued before the
// first digit is decided); another row is read with 16-byte global loads,
// four per thread in flight. pass(thr, f) calls f(key) for every key whose
// score is not -inf and whose order (the key's top 32 bits) is >= thr.
template <int kThreads>
struct RowSource {
  static constexpr int kBlock = kThreads * 4 * kUnroll;
  const float *row;
  int L;
  bool staged;
  float *stage;
  int chunk;            // scores per staged chunk
  uint32_t bar, phase;  // staging mbarrier and the parity of its next phase
  int resident, pending;
  volatile int *abort;

  // The score at or above which a key's order is >= thr: float_order is
  // monotonic, so one float compare replaces the order of every score (for
  // any finite score, order >= thr <=> score >= the returned value; no
  // finite score passes a NaN; -inf, the mark of an excluded key, never
  // passes).
  __device__ __forceinline__ static float threshold(uint32_t thr) {
    return (thr <= float_order(-3.402823466e38f)) ? -3.402823466e38f : order_float(thr);
  }
  template <class F>
  __device__ __forceinline__ static void key4(float4 v, long long i0, float tf, F &f) {
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e[q] >= tf)
        f((static_cast<uint64_t>(float_order(e[q])) << 32) |
          static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(i0 + q)));
    }
  }
  // Thread 0 starts copying chunk c (its 16-byte part; the tail of at most
  // three scores is read from global memory when processed).
  __device__ void issue(int c) {
    if (threadIdx.x == 0) {
      const long long c0 = static_cast<long long>(c) * chunk;
      const int n4 = static_cast<int>(min(static_cast<long long>(chunk), L - c0)) & ~3;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (n4 > 0) {
        ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n4) * 4u);
        ptx::bulk_g2s(ptx::smem_addr(stage), row + c0, static_cast<uint32_t>(n4) * 4u, bar);
      } else {
        ptx::mbar_arrive(bar);
      }
    }
    pending = c;
  }
  __device__ void prefetch() {
    if (staged && L > 0) issue(0);
  }
  __device__ void wait() {
    if (!ptx::mbar_wait(bar, phase, abort, 2000000000ull)) {
      volatile int no_abort = 0;   // give up on this row, but never leave with the copy in flight
      ptx::mbar_wait(bar, phase, &no_abort, 2000000000ull);
    }
    phase ^= 1u;
  }
  template <class F>
  __device__ void pass(uint32_t thr, F &&f) {
    const float tf = threshold(thr);
    if (!staged) {
      for (long long base = 0; base < L; base += kBlock) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const long long i0 = base + 4LL * (u * kThreads + threadIdx.x);
          v[u].x = (i0 + 0 < L) ? row[i0 + 0] : -INFINITY;
          v[u].y = (i0 + 1 < L) ? row[i0 + 1] : -INFINITY;
          v[u].z = (i0 + 2 < L) ? row[i0 + 2] : -INFINITY;
          v[u].w = (i0 + 3 < L) ? row[i0 + 3] : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) key4(v[u], base + 4LL * (u * kThreads + threadIdx.x), tf, f);
      }
      return;
    }
    const int nch = static_cast<int>((static_cast<long long>(L) + chunk - 1) / chunk);
    for (int c = 0; c < nch; ++c) {
      if (resident != c) {
        if (pending != c) {
          __syncthreads();   // everyone is done with the previous chunk
          issue(c);
        }
        wait();
        resident = c;
        pending = -1;
      }
      // (after a copy that never completed the chunk holds stale scores: the
      // pass goes on, every index stays bounded, and the call reports it)
      const long long c0 = static_cast<long long>(c) * chunk;
      const int n = static_cast<int>(min(static_cast<long long>(chunk), L - c0)), n4 = n & ~3;
      const float4 *s4 = reinterpret_cast<const float4 *>(stage);
      for (int i = threadIdx.x; i < (n4 >> 2); i += kThreads) key4(s4[i], c0 + 4LL * i, tf, f);
      for (int i = n4 + threadIdx.x; i < n; i += kThreads) {
        const float e = row[c0 + i];
        if (e >= tf)
          f((static_cast<uint64_t>(float_order(e)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(c0 + i)));
      }
    }
  }
};

// One warp sorts buf[start .. start+n) (n <= 32*E) descending in registers
// (E keys per lane, lane l holding positions l*E .. l*E+E-1; padding keys 0
// sort last) and hands each key with its final position to emit.
template <int E, class Emit>
__device__ __forceinline__ void warp_sort_segment(const uint64_t *buf, int start, int n, Emit &emit) {
  const int lane = threadIdx.x & 31;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = (lane * E + e < n) ? buf[start + lane * E + e] : 0ull;
  constexpr int m = 32 * E;
#pragma unroll
  for (int sz = 2; sz <= m; sz <<= 1) {
#pragma unroll
    for (int s = sz >> 1; s > 0; s >>= 1) {
      if (s < E) {  // both keys of a pair in this lane
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & s) == 0) {
            const bool desc = (((lane * E + e) & sz) == 0);
            if ((v[e] < v[e | s]) == desc) {
              const uint64_t x = v[e];
              v[e] = v[e | s];
              v[e | s] = x;
            }
          }
        }
      } else {      // partner in lane ^ (s / E)
        const int ls = s / E;
        const bool lower = (lane & ls) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t pv = __shfl_xor_sync(0xFFFFFFFFu, v[e], ls);
          const bool desc = (((lane * E + e) & sz) == 0);
          v[e] = (lower == desc) ? (v[e] > pv ? v[e] : pv) : (v[e] < pv ? v[e] : pv);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (lane * E + e < n) emit(v[e], start + lane * E + e);
}

// One warp orders buf[start .. start+n) (64 < n <= 256 keys of one first-digit
// bin) by splitting it on the next 8 key bits: a count of the keys per sub-bin
// (cnt: this warp's 256 counters in shared memory), a descending exclusive
// scan of the counts gives each sub-bin's start, the keys are scattered to
// their sub-bins, and each key's final rank is its sub-bin's start plus the
// number of keys of its sub-bin that are larger. Returns false, having
// written nothing, when some sub-bin holds more than 32 keys (many equal
// leading bits, e.g. tied scores): the caller then sorts the bin by
// comparisons.
template <class Emit>
__device__ __forceinline__ bool warp_radix_segment(uint64_t *buf, int start, int n, uint32_t *cnt, Emit &emit) {
  const int lane = threadIdx.x & 31;
  constexpr int E = 8;                       // keys per lane: key j = lane + 32 e
#pragma unroll
  for (int i = lane; i < 256; i += 32) cnt[i] = 0u;
  __syncwarp();
  uint64_t kk[E];
  uint32_t dg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    kk[e] = (j < n) ? buf[start + j] : 0ull;
    dg[e] = static_cast<uint32_t>(kk[e] >> 44) & 255u;
    if (j < n) atomicAdd(&cnt[dg[e]], 1u);
  }
  __syncwarp();
  // descending exclusive scan: lane owns digits 255 - 8 lane - u (u < 8)
  uint32_t c8[8], tot = 0, mx = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    c8[u] = cnt[255 - 8 * lane - u];
    tot += c8[u];
    mx = max(mx, c8[u]);
  }
  if (__reduce_max_sync(0xFFFFFFFFu, mx) > 32u) return false;
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  uint32_t r = incl - tot;
  __syncwarp();
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    cnt[255 - 8 * lane - u] = r | (c8[u] << 16);   // sub-bin start | its count
    r += c8[u];
  }
  __syncwarp();
  // scatter into the sub-bins (any order within one), then rank within each
  uint32_t cur[E];
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (lane + 32 * e < n) cur[e] = atomicAdd(&cnt[dg[e]], 1u) & 0xFFFFu;   // start + arrival order
  __syncwarp();
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (lane + 32 * e < n) buf[start + static_cast<int>(cur[e])] = kk[e];
  __syncwarp();
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (lane + 32 * e >= n) continue;
    const uint32_t sc = cnt[dg[e]];               // (start + count) | count << 16 after the arrivals
    const int c = static_cast<int>(sc >> 16);
    const int s0 = static_cast<int>(sc & 0xFFFFu) - c;
    int rank = 0;
    for (int x = s0; x < s0 + c; ++x) rank += (buf[start + x] > kk[e]) ? 1 : 0;
    emit(kk[e], start + s0 + rank);
  }
  __syncwarp();
  return true;
}

// Split collection, ahead of topk_stream_kernel on rows that come with the
// scorer's first-digit histogram: CTA c of row t takes the c-th slice of the
// row and appends every key the selection would place (at or above the
// boundary bin, or every key when the row holds at most k) to the row's
// candidate list. It decides from the histogram exactly as the selection
// does; rows the selection will refine are left alone. The selection checks
// the list's length against the histogram before it uses the list, and
// otherwise reads the row itself.
__global__ void __launch_bounds__(kCollectThreads) select_collect_kernel(ScoreParams p,
                                                                        const float *__restrict__ scores,
                                                                        long long ld,
                                                                        const uint32_t *__restrict__ hist,
                                                                        uint64_t *__restrict__ cand,
                                                                        uint32_t *__restrict__ cand_cnt, int cap) {
  constexpr int kW = kCollectThreads / 32, kPerC = kBins / kCollectThreads;
  constexpr int kRound = 4 * kCollectThreads;   // keys per round (one 16-byte load per thread)
  constexpr int kBatch = 8;                      // rounds whose loads are in flight together
  static_assert(kCollectBuf >= 2 * kRound, "a round never overfills the buffer");
  __shared__ uint32_t warp_sum[kW], warp_max[kW];
  __shared__ int s_bin, s_cnt;
  __shared__ uint32_t s_n, s_base;
  __shared__ uint64_t s_buf[kCollectBuf];
  const int t = blockIdx.y, c = blockIdx.x, C = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int L = p.valid_lens[t];
  if (bad_len(p, L) || L <= kSmallRow) return;
  const uint32_t k = static_cast<uint32_t>(p.top_k);
  const long long per = ((static_cast<long long>(L) + C - 1) / C + 3) & ~3LL;
  const long long s0 = static_cast<long long>(c) * per, s1 = min(static_cast<long long>(L), s0 + per);
  const float *row = scores + static_cast<long long>(t) * ld;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  // The slice's first kBatch rounds (one 16-byte load per thread and round)
  // are loaded before the boundary is decided: the two latencies overlap.
  auto load_batch = [&](long long base, float4 (&v)[kBatch]) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const long long i0 = base + static_cast<long long>(u) * kRound + 4LL * tid;
      if (vec && i0 + 3 < s1) {
        v[u] = __ldcs(reinterpret_cast<const float4 *>(row + i0));
      } else {
        v[u].x = (i0 + 0 < s1) ? row[i0 + 0] : -INFINITY;
        v[u].y = (i0 + 1 < s1) ? row[i0 + 1] : -INFINITY;
        v[u].z = (i0 + 2 < s1) ? row[i0 + 2] : -INFINITY;
        v[u].w = (i0 + 3 < s1) ? row[i0 + 3] : -INFINITY;
      }
    }
  };
  float4 v[kBatch];
  load_batch(s0, v);
  // descending scan of the first-digit histogram (thread tid: bins kBins-1-kPerC*tid-j)
  const uint32_t *h = hist + static_cast<size_t>(t) * kBins;
  uint32_t cnt[kPerC], tot = 0;
#pragma unroll
  for (int j = 0; j < kPerC; ++j) {
    cnt[j] = h[kBins - 1 - kPerC * tid - j];
    tot += cnt[j];
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  if (tid == 0) {
    s_bin = 0;
    s_cnt = 0;
  }
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    if (w < warp) before += warp_sum[w];
    all += warp_sum[w];
  }
  const bool take_all = all <= k;
  uint32_t run = before + incl - tot, mx = 0;
#pragma unroll
  for (int j = 0; j < kPerC; ++j) {
    if (!take_all && run < k && run + cnt[j] >= k) {
      s_bin = kBins - 1 - kPerC * tid - j;
      s_cnt = static_cast<int>(cnt[j]);
    }
    if (cnt[j] != 0u && (take_all || run + cnt[j] < k)) mx = max(mx, cnt[j]);   // bins above the boundary
    run += cnt[j];
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  if (lane == 0) warp_max[warp] = mx;
  __syncthreads();
  uint32_t max_above = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) max_above = max(max_above, warp_max[w]);
  if (max_above > static_cast<uint32_t>(kRankBinMax) || (!take_all && s_cnt > kBndCap)) return;
  const uint32_t thr = take_all ? 0u : static_cast<uint32_t>(s_bin);   // first digit of the weakest key taken

  uint64_t *out = cand + static_cast<size_t>(t) * cap;
  // Keys go to a shared-memory buffer first (one shared atomic per warp and
  // element position); the buffer goes out with one global reservation when
  // it holds a round's worth, and at the end.
  if (tid == 0) s_n = 0u;
  __syncthreads();
  auto flush = [&]() {   // all threads, after a barrier
    const uint32_t n = s_n;
    if (tid == 0) s_base = atomicAdd(cand_cnt + t, n);
    __syncthreads();
    const uint32_t b0 = s_base;
    for (uint32_t i = tid; i < n; i += kCollectThreads)
      if (b0 + i < static_cast<uint32_t>(cap)) out[b0 + i] = s_buf[i];
    __syncthreads();
    if (tid == 0) s_n = 0u;
    __syncthreads();
  };
  for (long long bb = s0; bb < s1; bb += static_cast<long long>(kBatch) * kRound) {
    if (bb != s0) load_batch(bb, v);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const long long base = bb + static_cast<long long>(u) * kRound;
      if (base >= s1) break;   // (uniform: every thread has the same base)
      const long long i0 = base + 4LL * tid;
      const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool ok = e[q] != -INFINITY && (float_order(e[q]) >> 20) >= thr;
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, ok);
        if (m == 0u) continue;
        uint32_t slot0 = 0;
        if (lane == 0) slot0 = atomicAdd(&s_n, static_cast<uint32_t>(__popc(m)));
        slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
        const uint32_t slot = slot0 + __popc(m & lanemask_lt());
        if (ok && slot < static_cast<uint32_t>(kCollectBuf)) s_buf[slot] = pack_key(e[q], static_cast<int32_t>(i0 + q));
      }
      __syncthreads();
      if (s_n > static_cast<uint32_t>(kCollectBuf - kRound)) flush();   // room for one more round
    }
  }
  __syncthreads();
  if (s_n > 0u) flush();
}

template <int kThreads, int kParts>
__global__ void __launch_bounds__(kThreads, 1024 / kThreads) topk_stream_kernel(ScoreParams p, const float *__restrict__ scores,
                                                              long long ld, const uint32_t *__restrict__ hist,
                                                              const uint64_t *__restrict__ cand,
                                                              uint32_t *__restrict__ cand_cnt, int cand_cap) {
  constexpr int kPer = kBins / kThreads;           // bins each thread owns in a scan
  // Bins up to kWarpBin keys are sorted by one warp in registers: 128 with
  // 1024 threads per row; 256 with 512 (more rows than SMs, as in prefill,
  // where broad selections fill many bins past 128 and a warp-sorted bin
  // saves the CTA-wide split).
  constexpr int kWarpBin = kThreads == 1024 ? 128 : 256;
  // Bins above kRadixMin keys are split on the next 8 bits rather than sorted
  // by comparisons (512 threads, where bins of 65..256 keys are common).
  constexpr int kRadixMin = kThreads == 1024 ? 128 : 64;
  constexpr int kLargeKeys = kBndCap / kThreads;   // a large bin's keys per thread
  static_assert(kBndCap % kThreads == 0 && kThreads <= kMaxThreads, "a large bin's keys spread evenly");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelShared *sh = reinterpret_cast<SelShared *>(smem_raw);
  const SelSmem lay = sel_smem(p.top_k, static_cast<long long>(p.max_lb) * p.epb);
  uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw + lay.buf);
  const int cap = static_cast<int>(lay.cap);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // With several CTAs a row (parts > 1: rows that leave SMs idle), all decide
  // the boundary alike, then CTA h places, orders and writes only the bins of
  // part h of the output: the bins whose buffer segment starts in
  // [h total / parts, (h + 1) total / parts). Whatever is not decided on the
  // first digit, and the padding, is the first CTA's.
  // (only the 1024-thread variant is launched so; one instantiation per count)
  constexpr int parts = kParts;
  static_assert(parts >= 1 && parts <= kMaxParts && (kThreads == 1024 || parts == 1), "parts");
  const int t = blockIdx.x / parts, h = blockIdx.x - t * parts;
  const int k = p.top_k;
  int32_t *oi = p.topk_idx + static_cast<long long>(t) * k;
  float *os = p.topk_score + static_cast<long long>(t) * k;
  // The row length is an input of the call, complete before the call's first
  // kernel (launched in plain stream order) started: read it at once, so the
  // row's copy can go out as soon as the scores are there.
  const int L = p.valid_lens[t];
  // This kernel may be launched before the one writing its input has ended:
  // wait for that kernel's completion and memory first.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // the first digit's counts
  uint32_t hpre[kPer];
  if (hist != nullptr) {
    const uint32_t *h = hist + static_cast<size_t>(t) * kBins;
#pragma unroll
    for (int j = 0; j < kPer; ++j) hpre[j] = h[kBins - 1 - kPer * tid - j];
  }
  if (bad_len(p, L)) {
    if (h != 0) return;
    if (tid == 0 && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_LEN);
    for (int i = tid; i < k; i += kThreads) {
      oi[i] = -1;
      os[i] = -INFINITY;
    }
    return;
  }
  const float *row = scores + static_cast<long long>(t) * ld;

  // ---- a short row: every candidate key into the buffer, one sort ----
  if (L <= kSmallRow && pow2_at_least(max(L, 64)) <= cap) {
    if (h != 0) return;
    if (tid == 0) sh->n_buf = 0;
    __syncthreads();
    for (int i = tid; i < L; i += kThreads) {
      const float v = row[i];
      if (v != -INFINITY) buf[atomicAdd(&sh->n_buf, 1)] = pack_key(v, i);   // at most L <= cap keys
    }
    __syncthreads();
    const int count = sh->n_buf;
    const int m = max(64, pow2_at_least(count));
    for (int i = count + tid; i < m; i += kThreads) buf[i] = 0ull;
    __syncthreads();
    sort_desc<kThreads>(buf, m);
    const int got = min(count, k);
    for (int i = tid; i < k; i += kThreads) {
      oi[i] = i < got ? key_index(buf[i]) : -1;
      os[i] = i < got ? key_score(buf[i]) : -INFINITY;
    }
    return;
  }

  const uint32_t sbar = ptx::smem_addr(smem_raw + lay.bar);
  RowSource<kThreads> rs{row, L, lay.stage_floats > 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0,
               reinterpret_cast<float *>(smem_raw + lay.stage), static_cast<int>(lay.stage_floats), sbar, 0u, -1, -1,
               &sh->abort_flag};
  if (tid == 0) {
    sh->abort_flag = 0;
    ptx::mbar_init(sbar, 1);
    ptx::fence_mbar_init();
  }
  if (cand == nullptr) rs.prefetch();   // the row is on its way while the first digit is decided
  if (tid == 0) {
    sh->b_bin = 0;
    sh->b_above = 0;
    sh->b_cnt = 0;
    sh->n_buf = 0;
    for (int q = 0; q < kMaxParts; ++q) sh->split_bin[q] = -1;
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
#pragma unroll
      for (int j = 0; j < kPer; ++j) c[j] = hpre[j];
    } else {
      for (int b = tid; b < kBins; b += kThreads) sh->table[b] = 0u;
      __syncthreads();
      rs.pass(0u, [&](uint64_t key) {
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
      // Also the largest such bin other than the boundary bin.
      uint32_t rb = run0, mx = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const bool rel = c[j] != 0u && rb < static_cast<uint32_t>(k);
        sh->table[kBins - 1 - kPer * tid - j] = rel ? (rb | (c[j] << 16)) : 0u;   // 0: holds none of the k best
        if (rel && (all <= static_cast<uint32_t>(k) || rb + c[j] < static_cast<uint32_t>(k))) mx = max(mx, c[j]);
        rb += c[j];
      }
      mx = __reduce_max_sync(0xFFFFFFFFu, mx);
      if (lane == 0) sh->warp_max[warp] = mx;
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

  uint32_t max_above = 0;   // largest first-digit bin above the boundary
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) max_above = max(max_above, sh->warp_max[w]);
  if (((take_all && rounds == 0) || (!take_all && rounds == 1)) && max_above <= kRankBinMax) {
    // ---- decided on the first digit: place, rank, write ----
    // (keys below the boundary bin are dropped on their top 32 bits alone)
    const int total = min(take_all ? static_cast<int>(all_keys) : sh->b_above + sh->b_cnt, cap);
    bool solo = parts == 1;
    if (!solo) {   // part q >= 1 starts at the highest bin whose segment starts at ceil(q total / parts) or later
      if (tid == 0) sh->n_large = 0;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const uint32_t e = sh->table[kBins - 1 - kPer * tid - j];
        if (e != 0u)
          for (int q = 1; q < parts; ++q)
            if ((e & 0xFFFFu) >= static_cast<uint32_t>((q * total + parts - 1) / parts))
              atomicMax(&sh->split_bin[q], kBins - 1 - kPer * tid - j);
        if (static_cast<int>(e >> 16) > kWarpBin) atomicAdd(&sh->n_large, 1);
      }
      __syncthreads();
      // so many large bins that the whole buffer is sorted at once: the first CTA alone
      solo = sh->n_large > kMaxLarge;
      if (solo && h != 0) return;
    }
    // bin b is this CTA's: at most split_bin[h] (part 0: any), above split_bin[h + 1] (last part: any)
    const int hi_bin = (h > 0) ? sh->split_bin[h] : kBins, lo_bin = (h + 1 < parts) ? sh->split_bin[h + 1] : -1;
    auto mine = [&](int b) { return solo || (b <= hi_bin && b > lo_bin); };
    auto place = [&](uint64_t key) {
      if ((key & mask) >= prefix && mine(static_cast<int>(key >> 52))) {
        const uint32_t old = atomicAdd(&sh->table[key >> 52], 1u);
        if (static_cast<int>(old & 0xFFFFu) < cap) buf[old & 0xFFFFu] = key;
      }
    };
    // the split collection's list, when it holds exactly the keys to place
    const uint32_t want = take_all ? all_keys : static_cast<uint32_t>(sh->b_above + sh->b_cnt);
    const uint32_t n_cand = (cand != nullptr) ? cand_cnt[t] : 0u;
    if (cand != nullptr && n_cand == want && n_cand <= static_cast<uint32_t>(cand_cap)) {
      const uint64_t *cl = cand + static_cast<size_t>(t) * cand_cap;
      for (int i = tid; i < static_cast<int>(n_cand); i += kThreads) place(cl[i]);
    } else {
      rs.pass(static_cast<uint32_t>(prefix >> 32), place);
    }
    __syncthreads();
    // Every bin holding some of the k best keys is now a contiguous segment
    // of buf. Bins of more than kWarpBin keys ("large") are first ordered by
    // the next 8 key bits, one bin at a time by the whole CTA, so each of
    // their keys is then ranked only among keys sharing those bits too; the
    // other bins are sorted by one warp each, in registers. Many large bins
    // (broad selections) make one bitonic sort of the whole buffer cheaper.
    if (tid == 0) sh->n_large = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t e = sh->table[kBins - 1 - kPer * tid - j];
      if (static_cast<int>(e >> 16) > kWarpBin && mine(kBins - 1 - kPer * tid - j)) {
        const int slot = atomicAdd(&sh->n_large, 1);
        if (slot < kMaxLarge) sh->large[slot] = e;
      }
    }
    __syncthreads();
    const int n_large = sh->n_large;
    if (n_large > kMaxLarge) {
      const int m = max(64, pow2_at_least(total));   // total <= k - 1 + kBndCap, m <= cap
      for (int i = total + tid; i < m; i += kThreads) buf[i] = 0ull;
      __syncthreads();
      sort_desc<kThreads>(buf, m);
      for (int i = tid; i < min(total, k); i += kThreads) emit(buf[i], i);
    } else {
      for (int x = 0; x < n_large; ++x) {
        const uint32_t e = sh->large[x];
        const int n = static_cast<int>(e >> 16);
        const int start = max(0, min(static_cast<int>(e & 0xFFFFu) - n, total));
        const int cnt = min(n, total - start);
        if (tid < 256) sh->sub_cnt[tid] = 0u;
        __syncthreads();
        uint64_t kk[kLargeKeys];   // this thread's keys of the bin
        uint32_t sd[kLargeKeys], sp[kLargeKeys];
#pragma unroll
        for (int u = 0; u < kLargeKeys; ++u) {
          const int q = tid + u * kThreads;
          kk[u] = (q < cnt) ? buf[start + q] : 0ull;
          sd[u] = static_cast<uint32_t>(kk[u] >> 44) & 255u;
          if (q < cnt) atomicAdd(&sh->sub_cnt[sd[u]], 1u);
        }
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
#pragma unroll
        for (int u = 0; u < kLargeKeys; ++u)
          if (tid + u * kThreads < cnt) sp[u] = atomicAdd(&sh->sub_cur[sd[u]], 1u);
        __syncthreads();   // the bin's keys are all in registers: its segment may be rewritten
#pragma unroll
        for (int u = 0; u < kLargeKeys; ++u)
          if (tid + u * kThreads < cnt) buf[start + static_cast<int>(sp[u])] = kk[u];
        __syncthreads();
        // sub_cur[d] now ends sub-bin d's run; it starts sub_cnt[d] earlier
#pragma unroll
        for (int u = 0; u < kLargeKeys; ++u) {
          if (tid + u * kThreads < cnt) {
            const int q1 = start + static_cast<int>(sh->sub_cur[sd[u]]), q0 = q1 - static_cast<int>(sh->sub_cnt[sd[u]]);
            int pos = q0;
            for (int q = q0; q < q1; ++q) pos += (buf[q] > kk[u]) ? 1 : 0;
            emit(kk[u], pos);
          }
        }
        __syncthreads();   // sub_cnt / sub_cur are reused by the next large bin
      }
      // Warp w orders the small bins w, w + 16, ... one at a time and writes
      // each key to its output slot: bins of up to kRadixMin keys by a sort in
      // registers, larger ones by a split on the next 8 key bits (in 256
      // counters per warp, in the row's staging area, which the place pass
      // is done with), or by a sort when that split leaves a crowded sub-bin.
      auto emit_if = [&](uint64_t kv, int pos) { emit(kv, pos); };
      uint32_t *radix_cnt = (lay.stage_floats >= static_cast<size_t>(kThreads / 32) * 256)
                                ? reinterpret_cast<uint32_t *>(smem_raw + lay.stage) + warp * 256
                                : nullptr;
      for (int b0 = warp; b0 < kBins; b0 += 32 * (kThreads / 32)) {
        const int b = b0 + (kThreads / 32) * lane;       // this lane's bin of the group
        const uint32_t pk = (b < kBins && mine(b)) ? sh->table[b] : 0u;
        uint32_t todo = __ballot_sync(0xFFFFFFFFu, pk != 0u && static_cast<int>(pk >> 16) <= kWarpBin);
        while (todo) {
          const int l = __ffs(todo) - 1;
          todo &= todo - 1;
          const uint32_t e = __shfl_sync(0xFFFFFFFFu, pk, l);
          const int n = static_cast<int>(e >> 16);
          const int start = max(0, min(static_cast<int>(e & 0xFFFFu) - n, total));   // the cursor ended at start + n
          const int cnt = min(n, total - start);
          if (cnt <= 32) warp_sort_segment<1>(buf, start, cnt, emit_if);
          else if (cnt <= 64) warp_sort_segment<2>(buf, start, cnt, emit_if);
          else if (cnt > kRadixMin && radix_cnt != nullptr && warp_radix_segment(buf, start, cnt, radix_cnt, emit_if)) {
          } else if (kWarpBin <= 128 || cnt <= 128) warp_sort_segment<4>(buf, start, cnt, emit_if);
          else if constexpr (kWarpBin > 128) warp_sort_segment<8>(buf, start, cnt, emit_if);
        }
      }
    }
    produced = min(total, k);
  } else {
    // ---- decided on a later digit, or a bin above the boundary too large to
    // rank by comparison: collect, sort, write ----
    if (h != 0) return;
    rs.pass(static_cast<uint32_t>(prefix >> 32), [&](uint64_t key) {
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
    sort_desc<kThreads>(buf, m);
    produced = min(count, k);
    for (int i = tid; i < produced; i += kThreads) emit(buf[i], i);
  }
  for (int i = produced + tid; h == 0 && i < k; i += kThreads) {
    oi[i] = -1;
    os[i] = -INFINITY;
  }
  if (tid == 0 && sh->abort_flag && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_TIMEOUT);
  if (cand_cnt != nullptr && parts == 1) {   // (with several CTAs a row the q preparation of the next call zeroes it)
    __syncthreads();   // every thread has read the row's count
    if (tid == 0) cand_cnt[t] = 0u;   // left zero for the next call
  }
}

}  // namespace

SelectPlan select_plan(int T, int top_k, long long max_len, bool have_scores_out, long long ld_out,
                       int split_sms) {
  SelectPlan pl{};
  pl.own_scores = !have_scores_out;
  pl.ld = have_scores_out ? ld_out : max_len;
  pl.scores_off = 0;
  pl.total = pl.own_scores ? ((static_cast<size_t>(T) * static_cast<size_t>(max_len) * 4 + 255) & ~size_t(255)) : 0;
  // Fewer rows than SMs, each long: split the collection so about two CTAs
  // per SM stream the rows, at least kCollectMin keys each. (On rows of up
  // to 32K keys the extra launch costs more than it saves: +10 us per call
  // on 64 rows of 8K-32K keys, against -25 us on 16 rows of 256K keys.)
  if (split_sms > 0 && T > 0 && T < split_sms && max_len >= kSplitMinLen) {
    const long long by_sms = (2LL * split_sms + T - 1) / T;
    const long long by_len = (max_len + kCollectMin - 1) / kCollectMin;
    const int chunks = static_cast<int>(std::min<long long>(std::min(by_sms, by_len), kMaxChunks));
    if (chunks >= 2) {
      pl.chunks = chunks;
      pl.cand_cap = static_cast<int>(sel_smem(top_k, max_len).cap);
      pl.cand_off = pl.total;
      pl.total += (static_cast<size_t>(T) * pl.cand_cap * 8 + 255) & ~size_t(255);
      pl.cnt_off = pl.total;
      pl.total += (static_cast<size_t>(T) * 4 + 255) & ~size_t(255);
    }
  }
  return pl;
}

bool select_supported(int top_k, long long max_len) {
  return sel_smem(top_k, max_len).total <= 227 * 1024;
}

cudaError_t launch_select(const ScoreParams &p, const float *scores, long long ld, const uint32_t *hist,
                          const SelectPlan &pl, void *workspace, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  const size_t smem = sel_smem(p.top_k, static_cast<long long>(p.max_lb) * p.epb).total;
  // One CTA per row: when every row gets an SM of its own and rows are longer
  // than a whole-row sort, 1024 threads; with more rows than SMs, 512 (two
  // CTAs share an SM when shared memory allows), and 512 for short rows, whose
  // single sort of at most kSmallRow keys gains nothing from more warps.
  const int sms = device_sm_count();
  const bool wide = sms > 0 && p.T <= sms && static_cast<long long>(p.max_lb) * p.epb > kSmallRow;
  uint64_t *cand = nullptr;
  uint32_t *cand_cnt = nullptr;
  if (pl.chunks > 0 && hist != nullptr) {
    cand = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(workspace) + pl.cand_off);
    cand_cnt = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(workspace) + pl.cnt_off);
  }
  // Rows that leave SMs idle: several CTAs a row (the 1024-thread variant), each
  // ordering and writing the bins of one part of the output; 2 when each streams
  // the whole row, up to kMaxParts when they read a collected candidate list.
  int parts = 1;
  if (wide)
    while (2 * parts <= (cand == nullptr ? 2 : kMaxParts) && 2 * parts * p.T <= sms) parts *= 2;
  void (*kern)(ScoreParams, const float *, long long, const uint32_t *, const uint64_t *, uint32_t *, int) =
      !wide ? topk_stream_kernel<512, 1>
            : parts == 4 ? topk_stream_kernel<1024, 4> : parts == 2 ? topk_stream_kernel<1024, 2> : topk_stream_kernel<1024, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (cand != nullptr) {
    cudaLaunchConfig_t ca{};
    ca.gridDim = dim3(static_cast<unsigned>(pl.chunks), static_cast<unsigned>(p.T), 1);
    ca.blockDim = dim3(kCollectThreads, 1, 1);
    ca.stream = stream;
    cudaLaunchAttribute aa[1];
    aa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    aa[0].val.programmaticStreamSerializationAllowed = 1;
    ca.attrs = aa;
    ca.numAttrs = 1;
    e = cudaLaunchKernelEx(&ca, select_collect_kernel, p, scores, ld, hist, cand, cand_cnt, pl.cand_cap);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.T * parts), 1, 1);
  cfg.blockDim = dim3(wide ? 1024 : 512, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the scorer's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, scores, ld, hist, static_cast<const uint64_t *>(cand),
                            cand_cnt, pl.cand_cap);
}

}  // namespace idx
