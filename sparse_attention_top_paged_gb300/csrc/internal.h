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
  const float *q, *w;
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
};

// Workspace sections of the tensor-core path (byte offsets; 256-aligned).
// In rows mode the scoring kernel writes every score to a [T, ld] matrix
// (`scores`, or the caller's scores_out) and the per-row top-k kernel selects;
// otherwise it keeps per-segment candidates for the merge kernel.
struct TcWorkspace {
  size_t seg_first, seg_last, cand_count, cand, scores, total;
  int num_ctas, n_slots;
  bool rows_mode;
  long long ld;  // row stride of the score matrix in rows mode
};

// Rows mode pays when a query keeps a large share of its keys (the streaming
// select inside the scoring kernel then compacts often): max_len < 8 * top_k.
bool tc_rows_mode(long long max_len, int top_k);
TcWorkspace tc_workspace_layout(int T, int top_k, int num_ctas, long long max_len, bool have_scores_out,
                                long long ld_scores_out);

// score_simt.cu
cudaError_t launch_score_simt(const ScoreParams &p, bool f32_keys, float *scores, long long ld,
                              cudaStream_t stream);
// topk.cu
cudaError_t launch_topk_rows(const ScoreParams &p, const float *scores, long long ld,
                             cudaStream_t stream);
cudaError_t launch_topk_merge(const ScoreParams &p, const TcWorkspace &ws, void *workspace,
                              cudaStream_t stream);
// score_tc.cu
bool score_tc_supported(const ScoreParams &p);
cudaError_t launch_score_tc(const ScoreParams &p, const TcWorkspace &ws, void *workspace,
                            cudaStream_t stream);  // rows mode: scores land in p.scores_out
// gather_pool.cu
cudaError_t launch_gather_kv(const idx_gather_kv_args &a, cudaStream_t stream);
cudaError_t launch_block_pool(const uint16_t *raw, const float *w, float *out, uint32_t first_block,
                              uint32_t n_new, uint32_t ratio, uint32_t hd, uint32_t rot, float theta,
                              float eps, cudaStream_t stream);
cudaError_t launch_expand_blocks(const int32_t *blocks, int T, int n_blocks, int ratio,
                                 int32_t *positions, cudaStream_t stream);
cudaError_t launch_valid_lens(const int32_t *block_lens, int T, int epb, int32_t *valid_lens,
                              cudaStream_t stream);

int device_sm_count();  // SMs of the current device (cached per device), 0 on error

}  // namespace idx
