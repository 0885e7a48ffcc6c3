// topk.cu — TopK(I[t,:], k) from a score matrix, on all SMs.
//
// Output order is the top-k write-out of "indexer_score_topk.cu": score
// descending, lower index first on equal scores, -1 / -inf padding. Both score
// paths write I[t, 0..valid_len) (with -inf for keys of out-of-range blocks)
// into a [T, ld] matrix; selection (BlockSelect, select.cuh) then runs in one
// of two plans:
//   * one pass: one CTA per query selects from its whole row and sorts the k
//     survivors (bitonic) — when a row fits one chunk;
//   * two stages: a grid of (chunk, query) CTAs each keeps the k best keys of
//     its chunk, then one CTA per query selects from that query's chunk
//     candidates and sorts — so long rows use every SM, not one per query.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace idx {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kBndCap = 2048;

__host__ __device__ inline int pow2_at_least(int k) {
  int kp = 1;
  while (kp < k) kp <<= 1;
  return kp;
}

// Shared memory of a selecting CTA: SelectShared, TopkShared, out (a power of
// two >= k keys), boundary buffer.
struct SelectSmem {
  size_t sel, tsh, out, bnd, total;
};

__host__ __device__ inline SelectSmem select_smem(int k) {
  SelectSmem m{};
  size_t off = 0;
  m.sel = off;
  off += (sizeof(SelectShared) + 15) & ~size_t(15);
  m.tsh = off;
  off += (sizeof(TopkShared) + 15) & ~size_t(15);
  m.out = off;
  off += static_cast<size_t>(pow2_at_least(k)) * 8;
  m.bnd = off;
  off += static_cast<size_t>(kBndCap) * 8;
  m.total = off;
  return m;
}

__device__ __forceinline__ BlockSelect<kTopkThreads> make_select(unsigned char *smem, int k) {
  const SelectSmem m = select_smem(k);
  return BlockSelect<kTopkThreads>{reinterpret_cast<SelectShared *>(smem + m.sel),
                                   reinterpret_cast<TopkShared *>(smem + m.tsh),
                                   reinterpret_cast<uint64_t *>(smem + m.out),
                                   reinterpret_cast<uint64_t *>(smem + m.bnd), kBndCap, 1};
}

__device__ __forceinline__ bool bad_len(const ScoreParams &p, int L) {
  return L < 0 || static_cast<long long>(L) > static_cast<long long>(p.max_lb) * p.epb;
}

__device__ void write_padding(const ScoreParams &p, int t) {
  if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_LEN);
  for (int i = threadIdx.x; i < p.top_k; i += kTopkThreads) {
    p.topk_idx[static_cast<long long>(t) * p.top_k + i] = -1;
    p.topk_score[static_cast<long long>(t) * p.top_k + i] = -INFINITY;
  }
}

__device__ void write_sorted(const ScoreParams &p, int t, BlockSelect<kTopkThreads> &sel, int count) {
  const int k = p.top_k;
  sel.sort_desc(count);
  int32_t *out_i = p.topk_idx + static_cast<long long>(t) * k;
  float *out_s = p.topk_score + static_cast<long long>(t) * k;
  for (int i = threadIdx.x; i < k; i += kTopkThreads) {
    if (i < count) {
      const uint64_t key = sel.out[i];
      out_i[i] = key_index(key);
      out_s[i] = key_score(key);
    } else {
      out_i[i] = -1;
      out_s[i] = -INFINITY;
    }
  }
}

// Scores row[lo .. lo+n) as keys (index = position in the row; -inf = none).
struct RowSrc {
  const float *row;
  int lo;
  __device__ void begin() {}
  __device__ __forceinline__ uint64_t get(int i) const {
    const float v = row[lo + i];
    return v == -INFINITY ? 0ull : pack_key(v, lo + i);
  }
};

// The candidates of chunks j0 .. j0+nseg-1 laid end to end (offsets in seg_off).
struct CandSrc {
  const uint64_t *cand;
  const int *seg_off;
  long long j0;
  int k, js;
  __device__ void begin() { js = 0; }
  __device__ __forceinline__ uint64_t get(int i) {
    while (seg_off[js + 1] <= i) ++js;   // i increases per thread within a pass
    return cand[(j0 + js) * k + (i - seg_off[js])];
  }
};

// ---------------------------------------------------------------- one pass --
__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(ScoreParams p, const float *scores, long long ld) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int t = blockIdx.x;
  const int L = p.valid_lens[t];
  if (bad_len(p, L)) return write_padding(p, t);
  BlockSelect<kTopkThreads> sel = make_select(smem_raw, p.top_k);
  RowSrc src{scores + static_cast<long long>(t) * ld, 0};
  const int count = sel.run(src, L, p.top_k);
  write_sorted(p, t, sel, count);
}

// ------------------------------------------------------ stage 1: chunks ----
__global__ void __launch_bounds__(kTopkThreads) topk_chunk_kernel(ScoreParams p, const float *scores, long long ld,
                                                                  int chunk, int n_ch, uint64_t *cand,
                                                                  int32_t *cand_count) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int c = blockIdx.x, t = blockIdx.y;
  const long long slot = static_cast<long long>(t) * n_ch + c;
  const int L = p.valid_lens[t];
  const int lo = c * chunk;
  const int hi = bad_len(p, L) ? lo : min(L, lo + chunk);
  if (hi <= lo) {
    if (threadIdx.x == 0) cand_count[slot] = 0;
    return;
  }
  BlockSelect<kTopkThreads> sel = make_select(smem_raw, p.top_k);
  RowSrc src{scores + static_cast<long long>(t) * ld, lo};
  const int count = sel.run(src, hi - lo, p.top_k);
  uint64_t *dst = cand + slot * p.top_k;
  for (int i = threadIdx.x; i < count; i += kTopkThreads) dst[i] = sel.out[i];
  if (threadIdx.x == 0) cand_count[slot] = count;
}

// ------------------------------------------------------- stage 2: merge ----
__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(ScoreParams p, int n_ch, const uint64_t *cand,
                                                                  const int32_t *cand_count) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int warp_tot[kTopkThreads / 32];
  const int t = blockIdx.x;
  const int L = p.valid_lens[t];
  if (bad_len(p, L)) return write_padding(p, t);
  // chunk offsets (prefix of the counts) live behind the selection's own memory
  int *seg_off = reinterpret_cast<int *>(smem_raw + select_smem(p.top_k).total);
  const long long j0 = static_cast<long long>(t) * n_ch;
  int carry = 0;
  for (int cb = 0; cb < n_ch; cb += kTopkThreads) {
    const int j = cb + static_cast<int>(threadIdx.x);
    int cnt = (j < n_ch) ? cand_count[j0 + j] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, cnt, o);
      if (lane_id() >= static_cast<uint32_t>(o)) cnt += v;
    }
    if (lane_id() == 31) warp_tot[threadIdx.x >> 5] = cnt;
    __syncthreads();
    int before = carry;
    int all = 0;
    for (int wi = 0; wi < kTopkThreads / 32; ++wi) {
      if (wi < static_cast<int>(threadIdx.x >> 5)) before += warp_tot[wi];
      all += warp_tot[wi];
    }
    if (j < n_ch) seg_off[j + 1] = before + cnt;
    __syncthreads();
    carry += all;
  }
  if (threadIdx.x == 0) seg_off[0] = 0;
  __syncthreads();
  BlockSelect<kTopkThreads> sel = make_select(smem_raw, p.top_k);
  CandSrc src{cand, seg_off, j0, p.top_k, 0};
  const int count = sel.run(src, seg_off[n_ch], p.top_k);
  write_sorted(p, t, sel, count);
}

}  // namespace

SelectPlan select_plan(int T, int top_k, long long max_len, bool have_scores_out, long long ld_out) {
  SelectPlan pl{};
  const int kp = pow2_at_least(top_k);
  long long chunk = 16LL * kp;
  if (chunk < 4096) chunk = 4096;
  pl.chunk = static_cast<int>(chunk);
  pl.two_stage = max_len > chunk;
  pl.n_ch = pl.two_stage ? static_cast<int>((max_len + chunk - 1) / chunk) : 0;
  pl.own_scores = !have_scores_out;
  pl.ld = have_scores_out ? ld_out : max_len;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  pl.scores_off = off;
  if (pl.own_scores) off = al(off + static_cast<size_t>(T) * static_cast<size_t>(max_len) * 4);
  pl.count_off = off;
  if (pl.two_stage) off = al(off + static_cast<size_t>(T) * pl.n_ch * 4);
  pl.cand_off = off;
  if (pl.two_stage) off = al(off + static_cast<size_t>(T) * pl.n_ch * top_k * 8);
  pl.total = off;
  return pl;
}

bool select_supported(int top_k, long long max_len) {
  const long long chunk = 16LL * pow2_at_least(top_k) < 4096 ? 4096 : 16LL * pow2_at_least(top_k);
  const long long n_ch = max_len > chunk ? (max_len + chunk - 1) / chunk : 0;
  const size_t merge_smem = select_smem(top_k).total + static_cast<size_t>(n_ch + 1) * 4;
  return merge_smem <= 227 * 1024;
}

cudaError_t launch_select(const ScoreParams &p, const float *scores, long long ld, const SelectPlan &pl,
                          void *workspace, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  cudaError_t e;
  const size_t smem = select_smem(p.top_k).total;
  if (!pl.two_stage) {
    if ((e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
      return e;
    topk_rows_kernel<<<p.T, kTopkThreads, smem, stream>>>(p, scores, ld);
    return cudaGetLastError();
  }
  unsigned char *base = static_cast<unsigned char *>(workspace);
  uint64_t *cand = reinterpret_cast<uint64_t *>(base + pl.cand_off);
  int32_t *count = reinterpret_cast<int32_t *>(base + pl.count_off);
  if ((e = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return e;
  topk_chunk_kernel<<<dim3(pl.n_ch, p.T), kTopkThreads, smem, stream>>>(p, scores, ld, pl.chunk, pl.n_ch, cand,
                                                                      count);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t smem2 = smem + static_cast<size_t>(pl.n_ch + 1) * 4;
  if ((e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem2))) != cudaSuccess)
    return e;
  topk_merge_kernel<<<p.T, kTopkThreads, smem2, stream>>>(p, pl.n_ch, cand, count);
  return cudaGetLastError();
}

}  // namespace idx
