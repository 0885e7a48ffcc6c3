// topk.cu — per-query top-k selection and ordering.
//
// TopK(I[t,:], k) with the output order of the top-k write-out in
// "indexer_score_topk.cu" (score descending, lower index first on equal
// scores, -1 / -inf padding). One CTA per query streams its candidates
// through a shared-memory TopkGroup (threshold filter + in-place radix select,
// see common.cuh) and finishes with a bitonic sort of the k survivors. Two
// sources feed it:
//   * rows:  a full score row I[t, 0..valid_len) (CUDA-core path);
//   * merge: the per-segment candidate lists the tensor-core score kernel
//            wrote to the workspace (each already the top-k of its segment).
#include "common.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kFlatSegs = kTopkThreads;  // segments per query read in one flat pass

template <bool kMerge>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(ScoreParams p, const float *scores,
                                                            long long ld, const int32_t *seg_first,
                                                            const int32_t *seg_last,
                                                            const int32_t *cand_count,
                                                            const uint64_t *cand, int cap) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkShared *sh = reinterpret_cast<TopkShared *>(smem_raw);
  uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw + ((sizeof(TopkShared) + 15) & ~size_t(15)));
  const int t = blockIdx.x;
  const int k = p.top_k;
  const int L = p.valid_lens[t];
  int32_t *out_i = p.topk_idx + static_cast<long long>(t) * k;
  float *out_s = p.topk_score + static_cast<long long>(t) * k;

  if (L < 0 || static_cast<long long>(L) > static_cast<long long>(p.max_lb) * p.epb) {
    if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_LEN);
    for (int i = threadIdx.x; i < k; i += kTopkThreads) {
      out_i[i] = -1;
      out_s[i] = -INFINITY;
    }
    return;
  }

  TopkGroup<kTopkThreads> g{sh, buf, cap, static_cast<int>(threadIdx.x), 1};
  g.reset();
  if constexpr (!kMerge) {
    const float *row = scores + static_cast<long long>(t) * ld;
    for (int base = 0; base < L; base += kTopkThreads) {
      const int s = base + threadIdx.x;
      float v = -INFINITY;
      if (s < L) v = row[s];
      g.offer(pack_key(v, s), s < L && v != -INFINITY);
      g.after_round(k);
    }
  } else if (L > 0) {
    // The query's segments are slots j0..j1. With at most kFlatSegs of them,
    // read every count at once, prefix them in shared memory and stream all
    // candidates as one flat list (no per-segment round trip to memory).
    __shared__ int seg_off[kFlatSegs + 1];
    __shared__ int warp_tot[kTopkThreads / 32];
    const int j0 = seg_first[t], j1 = seg_last[t];
    const int nseg = j1 - j0 + 1;
    if (nseg <= kFlatSegs) {
      const int j = static_cast<int>(threadIdx.x);
      int c = (j < nseg) ? cand_count[j0 + j] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, c, o);
        if (lane_id() >= static_cast<uint32_t>(o)) c += v;
      }
      if (lane_id() == 31) warp_tot[threadIdx.x >> 5] = c;
      __syncthreads();
      int before = 0;
      for (int wi = 0; wi < static_cast<int>(threadIdx.x >> 5); ++wi) before += warp_tot[wi];
      if (j < nseg) seg_off[j + 1] = before + c;
      if (j == 0) seg_off[0] = 0;
      __syncthreads();
      const int total = seg_off[nseg];
      int js = 0;
      for (int base = 0; base < total; base += kTopkThreads) {
        const int i = base + static_cast<int>(threadIdx.x);
        const bool have = i < total;
        uint64_t key = 0ull;
        if (have) {
          while (seg_off[js + 1] <= i) ++js;   // segment holding flat index i (monotone in i)
          key = cand[static_cast<long long>(j0 + js) * k + (i - seg_off[js])];
        }
        g.offer(key, have);
        g.after_round(k);
      }
    } else {
      for (int j = j0; j <= j1; ++j) {
        const int n = cand_count[j];
        const uint64_t *c = cand + static_cast<long long>(j) * k;
        for (int base = 0; base < n; base += kTopkThreads) {
          const int i = base + threadIdx.x;
          const uint64_t key = (i < n) ? c[i] : 0ull;
          g.offer(key, i < n);
          g.after_round(k);
        }
      }
    }
  }
  g.compact(k);
  g.sort_desc();
  const int n = sh->count;
  for (int i = threadIdx.x; i < k; i += kTopkThreads) {
    if (i < n) {
      const uint64_t key = buf[i];
      out_i[i] = key_index(key);
      out_s[i] = key_score(key);
    } else {
      out_i[i] = -1;
      out_s[i] = -INFINITY;
    }
  }
}

size_t topk_smem(int k) {
  const int cap = topk_rows_cap(k, kTopkThreads);
  return ((sizeof(TopkShared) + 15) & ~size_t(15)) + static_cast<size_t>(cap) * 8;
}

template <bool kMerge>
cudaError_t launch(const ScoreParams &p, const float *scores, long long ld, const int32_t *sf,
                   const int32_t *sl, const int32_t *cc, const uint64_t *cand, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  const size_t smem = topk_smem(p.top_k);
  auto kern = topk_kernel<kMerge>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<p.T, kTopkThreads, smem, stream>>>(p, scores, ld, sf, sl, cc, cand,
                                            topk_rows_cap(p.top_k, kTopkThreads));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_rows(const ScoreParams &p, const float *scores, long long ld,
                             cudaStream_t stream) {
  return launch<false>(p, scores, ld, nullptr, nullptr, nullptr, nullptr, stream);
}

cudaError_t launch_topk_merge(const ScoreParams &p, const TcWorkspace &ws, void *workspace,
                              cudaStream_t stream) {
  unsigned char *base = static_cast<unsigned char *>(workspace);
  return launch<true>(p, nullptr, 0, reinterpret_cast<const int32_t *>(base + ws.seg_first),
                      reinterpret_cast<const int32_t *>(base + ws.seg_last),
                      reinterpret_cast<const int32_t *>(base + ws.cand_count),
                      reinterpret_cast<const uint64_t *>(base + ws.cand), stream);
}

}  // namespace idx
