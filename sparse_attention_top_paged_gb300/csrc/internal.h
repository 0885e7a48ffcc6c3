// internal.h — host-side interfaces between the libidx translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/idx.h"

namespace idx {

constexpr int kMaxTopK = 4096;

// Plain-data copy of the score arguments handed to kernels by value.
struct ScoreParams {
  int T, H, D;
  const float *q, *w;          // q: float32 queries (null when q16 is given)
  const uint16_t *q16;         // bf16 queries (tensor path), or null
  const uint8_t *keys_fp4, *key_scale;
  const float *key_gscale, *keys_f32;
  int P, epb;
  const int32_t *block_table;
  int max_lb;
  long long bt_stride;
  const int32_t *valid_lens;
  int top_k;
  int32_t *topk_idx;
  float *topk_score;
  float *scores_out;
  long long ld_scores;
  int32_t *dev_status;
  int q_format;   // idx_q_format_t
};

// How TopK(I[t,:], k) is taken from the [T, ld] score matrix: one streaming
// selection kernel per call; the workspace holds the matrix when the caller
// passes no scores_out (byte offsets; 256-aligned).
struct SelectPlan {
  bool own_scores;   // the score matrix lives in the workspace (no caller scores_out)
  long long ld;      // row stride of the score matrix
  size_t scores_off, total;
  // Split collection (few long rows next to a scorer histogram): `chunks` CTAs
  // per row gather the row's candidate keys into the workspace before the
  // one-CTA-per-row selection orders them. chunks == 0: no split.
  int chunks;
  int cand_cap;             // candidate keys per row
  size_t cand_off, cnt_off; // [T][cand_cap] composite keys, [T] counters (left zero)
};

// split_sms: SM count when the rows come with a scorer histogram (tensor
// path), 0 otherwise.
SelectPlan select_plan(int T, int top_k, long long max_len, bool have_scores_out, long long ld_out,
                       int split_sms);
bool select_supported(int top_k, long long max_len);  // the selection's buffers fit shared memory

// score_simt.cu
cudaError_t launch_score_simt(const ScoreParams &p, bool f32_keys, float *scores, long long ld,
                              cudaStream_t stream);
// topk.cu
// hist: per-query histograms of the top 12 key bits of the scores (from the
// tensor scorer), or nullptr.
cudaError_t launch_select(const ScoreParams &p, const float *scores, long long ld, const uint32_t *hist,
                          const SelectPlan &plan, void *workspace, cudaStream_t stream);
// score_tc.cu
bool score_tc_supported(const ScoreParams &p);
size_t score_tc_workspace(const ScoreParams &p);  // per-query q records (bytes)
// Also fills hist[t][d] (kScoreBins per query) with the number of valid keys
// of query t whose selection key has top 12 bits d, and zeroes cand_cnt[t]
// (the split collection's candidate counters) when cand_cnt is given.
constexpr int kScoreBins = 4096;
cudaError_t launch_score_tc(const ScoreParams &p, int num_ctas, void *qrec, uint32_t *hist, uint32_t *cand_cnt,
                            float *scores, long long ld, cudaStream_t stream);
// The NVFP4 query quantisation of the NVFP4-q mode, for `rows` head rows of 128.
cudaError_t launch_quantize_q_nvfp4(const float *q, long long rows, uint8_t *codes, uint8_t *scales, float *gscale,
                                    cudaStream_t stream);
// gather_pool.cu
cudaError_t launch_gather_kv(const idx_gather_kv_args &a, cudaStream_t stream);
cudaError_t launch_block_pool(const uint16_t *raw, const float *w, float *out, uint32_t first_block,
                              uint32_t n_new, uint32_t ratio, uint32_t hd, uint32_t rot, float theta,
                              float eps, cudaStream_t stream);
cudaError_t launch_qsa_qprep(const uint16_t *qk, const float *w, float *q_out, uint32_t rows, uint32_t first_pos,
                             uint32_t qkw, uint32_t n_heads, uint32_t hd, uint32_t rot, float theta, float eps,
                             cudaStream_t stream);
cudaError_t launch_expand_blocks(const int32_t *blocks, int T, int n_blocks, int ratio,
                                 int32_t *positions, cudaStream_t stream);
cudaError_t launch_valid_lens(const int32_t *block_lens, int T, int epb, int32_t *valid_lens,
                              cudaStream_t stream);

int device_sm_count();  // SMs of the current device (cached per device), 0 on error

}  // namespace idx
