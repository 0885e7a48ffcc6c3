// api.cu — the extern "C" entry points of libidx: host-side validation,
// workspace layout and dispatch to the kernels. See include/idx.h for the
// contract of each call.
#include <mutex>
#include <vector>

#include "internal.h"

namespace idx {

int device_sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace idx

using namespace idx;

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

enum class Plan { kNone, kSimt, kTensor };

struct Resolved {
  Plan plan = Plan::kNone;
  ScoreParams p{};
  size_t ws_bytes = 0;
  SelectPlan sel{};
  size_t qrec_off = 0, hist_off = 0;
  int num_ctas = 0;
};

idx_status_t resolve(const idx_score_topk_args *a, Resolved *r) {
  if (!a || !r) return IDX_ERR_INVALID_ARG;
  if (a->T < 0 || a->H < 1 || a->H > 256 || a->P < 1 || a->entries_per_block < 1 ||
      a->max_logical_blocks < 1 || a->bt_stride < 0 || a->top_k < 1 || a->top_k > kMaxTopK)
    return IDX_ERR_INVALID_ARG;
  if (a->key_format != IDX_KEYS_NVFP4 && a->key_format != IDX_KEYS_F32) return IDX_ERR_INVALID_ARG;
  if (a->path != IDX_PATH_AUTO && a->path != IDX_PATH_TENSOR && a->path != IDX_PATH_SIMT)
    return IDX_ERR_INVALID_ARG;
  if (a->num_ctas < 0) return IDX_ERR_INVALID_ARG;
  if (a->q_format != IDX_Q_EXACT && a->q_format != IDX_Q_NVFP4) return IDX_ERR_INVALID_ARG;
  if (a->q_dtype != IDX_Q_F32 && a->q_dtype != IDX_Q_BF16) return IDX_ERR_INVALID_ARG;
  const long long max_len = static_cast<long long>(a->max_logical_blocks) * a->entries_per_block;
  if (max_len > 0x7FFFFFFFLL) return IDX_ERR_INVALID_ARG;
  const bool f32 = a->key_format == IDX_KEYS_F32;
  if (f32) {
    if (a->D != 64 && a->D != 128) return IDX_ERR_UNSUPPORTED;
  } else {
    if (a->D != 128) return IDX_ERR_UNSUPPORTED;
    if (a->entries_per_block % 16 != 0) return IDX_ERR_UNSUPPORTED;
  }
  if (a->T > 0) {
    if (!a->q || !a->w || !a->block_table || !a->valid_lens || !a->topk_idx || !a->topk_score)
      return IDX_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->w, 4) || !aligned(a->block_table, 4) ||
        !aligned(a->valid_lens, 4) || !aligned(a->topk_idx, 4) || !aligned(a->topk_score, 4))
      return IDX_ERR_INVALID_ARG;
    if (f32) {
      if (!a->keys_f32 || !aligned(a->keys_f32, 16)) return IDX_ERR_INVALID_ARG;
    } else {
      if (!a->keys_fp4 || !a->key_scale || !a->key_gscale) return IDX_ERR_INVALID_ARG;
      if (!aligned(a->keys_fp4, 16) || !aligned(a->key_scale, 16) || !aligned(a->key_gscale, 4))
        return IDX_ERR_INVALID_ARG;
    }
    if (a->dev_status && !aligned(a->dev_status, 4)) return IDX_ERR_INVALID_ARG;
  }
  if (a->scores_out) {
    if (a->ld_scores < max_len || !aligned(a->scores_out, 4)) return IDX_ERR_INVALID_ARG;
  }

  Plan plan;
  if (a->path == IDX_PATH_SIMT)
    plan = Plan::kSimt;
  else if (a->path == IDX_PATH_TENSOR)
    plan = Plan::kTensor;
  else
    plan = f32 ? Plan::kSimt : Plan::kTensor;
  if (plan == Plan::kTensor && f32) return IDX_ERR_UNSUPPORTED;
  const bool nvfp4_q = a->q_format == IDX_Q_NVFP4;
  if (nvfp4_q && (plan != Plan::kTensor || a->H > 128)) return IDX_ERR_UNSUPPORTED;
  const bool bf16_q = a->q_dtype == IDX_Q_BF16;
  if (bf16_q && plan != Plan::kTensor) return IDX_ERR_UNSUPPORTED;

  ScoreParams &p = r->p;
  p.T = a->T; p.H = a->H; p.D = a->D;
  p.q = bf16_q ? nullptr : static_cast<const float *>(a->q);
  p.q16 = bf16_q ? static_cast<const uint16_t *>(a->q) : nullptr;
  p.w = a->w;
  p.keys_fp4 = a->keys_fp4; p.key_scale = a->key_scale;
  p.key_gscale = a->key_gscale; p.keys_f32 = a->keys_f32;
  p.P = a->P; p.epb = a->entries_per_block;
  p.block_table = a->block_table; p.max_lb = a->max_logical_blocks; p.bt_stride = a->bt_stride;
  p.valid_lens = a->valid_lens; p.top_k = a->top_k;
  p.topk_idx = a->topk_idx; p.topk_score = a->topk_score;
  p.scores_out = a->scores_out; p.ld_scores = a->ld_scores;
  p.dev_status = a->dev_status;
  p.q_format = a->q_format;

  if (plan == Plan::kTensor && !score_tc_supported(p)) {
    // (the NVFP4 q mode has no CUDA-core counterpart: never a silent fallback)
    if (a->path == IDX_PATH_TENSOR || nvfp4_q || bf16_q) return IDX_ERR_UNSUPPORTED;
    plan = Plan::kSimt;
  }
  r->plan = plan;
  if (plan == Plan::kTensor) {
    int g = a->num_ctas;
    if (g == 0) g = device_sm_count();
    if (g <= 0) return IDX_ERR_CUDA;
    r->num_ctas = g;
  }
  // Both paths write I[t, s] to a [T, ld] matrix (the caller's scores_out, or
  // the workspace), then select from it.
  if (!select_supported(a->top_k, max_len)) return IDX_ERR_UNSUPPORTED;
  r->sel = select_plan(a->T, a->top_k, max_len, a->scores_out != nullptr, a->ld_scores,
                       plan == Plan::kTensor ? device_sm_count() : 0);
  r->ws_bytes = r->sel.total;
  if (plan == Plan::kTensor) {  // then the scorer's per-query q records and key histograms
    r->qrec_off = r->ws_bytes;
    r->ws_bytes += (score_tc_workspace(p) + 255) & ~size_t(255);
    r->hist_off = r->ws_bytes;
    r->ws_bytes += static_cast<size_t>(a->T) * kScoreBins * 4;
  }
  return IDX_OK;
}

}  // namespace

extern "C" {

idx_status_t idx_score_topk_workspace_size(const idx_score_topk_args *args, size_t *bytes) {
  if (!bytes) return IDX_ERR_INVALID_ARG;
  Resolved r;
  const idx_status_t st = resolve(args, &r);
  if (st != IDX_OK) return st;
  *bytes = r.ws_bytes;
  return IDX_OK;
}

idx_status_t idx_score_topk(const idx_score_topk_args *args, idx_stream_t stream) {
  Resolved r;
  idx_status_t st = resolve(args, &r);
  if (st != IDX_OK) return st;
  if (args->T == 0) return IDX_OK;
  if (r.ws_bytes > 0) {
    if (!args->workspace || !aligned(args->workspace, 256)) return IDX_ERR_INVALID_ARG;
    if (args->workspace_bytes < r.ws_bytes) return IDX_ERR_WORKSPACE_TOO_SMALL;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t ev0 = static_cast<cudaEvent_t>(args->timing_events[0]);
  cudaEvent_t ev1 = static_cast<cudaEvent_t>(args->timing_events[1]);
  const bool timed = ev0 != nullptr && ev1 != nullptr;
  cudaError_t e = timed ? cudaEventRecord(ev0, s) : cudaSuccess;
  if (e != cudaSuccess) return IDX_ERR_CUDA;
  float *scores = r.sel.own_scores ? reinterpret_cast<float *>(static_cast<unsigned char *>(args->workspace) +
                                                               r.sel.scores_off)
                                   : args->scores_out;
  if (r.plan == Plan::kSimt)
    e = launch_score_simt(r.p, args->key_format == IDX_KEYS_F32, scores, r.sel.ld, s);
  else
    e = launch_score_tc(r.p, r.num_ctas, static_cast<unsigned char *>(args->workspace) + r.qrec_off,
                        reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(args->workspace) + r.hist_off),
                        r.sel.chunks > 0
                            ? reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(args->workspace) + r.sel.cnt_off)
                            : nullptr,
                        scores, r.sel.ld, s);
  if (e == cudaSuccess && timed) e = cudaEventRecord(ev1, s);
  const uint32_t *hist = r.plan == Plan::kTensor
                             ? reinterpret_cast<const uint32_t *>(static_cast<unsigned char *>(args->workspace) +
                                                                  r.hist_off)
                             : nullptr;
  if (e == cudaSuccess) e = launch_select(r.p, scores, r.sel.ld, hist, r.sel, args->workspace, s);
  return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

idx_status_t idx_quantize_q_nvfp4(const float *q, int64_t rows, uint8_t *codes, uint8_t *scales, float *gscale,
                                  idx_stream_t stream) {
  if (rows < 0) return IDX_ERR_INVALID_ARG;
  if (rows == 0) return IDX_OK;
  if (!q || !codes || !scales || !gscale || !aligned(q, 16) || !aligned(codes, 2) || !aligned(gscale, 4))
    return IDX_ERR_INVALID_ARG;
  return launch_quantize_q_nvfp4(q, rows, codes, scales, gscale, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? IDX_OK
             : IDX_ERR_CUDA;
}

idx_status_t idx_gather_kv(const idx_gather_kv_args *a, idx_stream_t stream) {
  if (!a) return IDX_ERR_INVALID_ARG;
  if (a->T < 0 || a->n_sel < 0 || a->max_logical_blocks < 1 || a->bt_stride < 0 || a->P < 1 ||
      a->block_size < 1 || a->row_bytes <= 0 || a->row_bytes % 16 != 0)
    return IDX_ERR_INVALID_ARG;
  if ((a->v_cache == nullptr) != (a->v_out == nullptr)) return IDX_ERR_INVALID_ARG;
  if (static_cast<long long>(a->T) * a->n_sel == 0) return IDX_OK;
  if (!a->sel || !a->block_table || !a->k_cache || !a->k_out) return IDX_ERR_INVALID_ARG;
  if (!aligned(a->k_cache, 16) || !aligned(a->k_out, 16) || !aligned(a->sel, 4) ||
      !aligned(a->block_table, 4))
    return IDX_ERR_INVALID_ARG;
  if (a->v_cache && (!aligned(a->v_cache, 16) || !aligned(a->v_out, 16))) return IDX_ERR_INVALID_ARG;
  if (a->dev_status && !aligned(a->dev_status, 4)) return IDX_ERR_INVALID_ARG;
  if ((static_cast<long long>(a->T) * a->n_sel + 7) / 8 > 0x7FFFFFFFLL) return IDX_ERR_UNSUPPORTED;
  return launch_gather_kv(*a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? IDX_OK
                                                                                      : IDX_ERR_CUDA;
}

idx_status_t idx_block_pool(const uint16_t *raw_keys, const float *k_norm_w, float *block_keys,
                            uint32_t first_block, uint32_t n_new, uint32_t ratio, uint32_t hd,
                            uint32_t rot, float theta, float eps, idx_stream_t stream) {
  if (hd < 32 || hd > 1024 || hd % 32 != 0 || rot % 2 != 0 || rot > hd || ratio < 1)
    return IDX_ERR_INVALID_ARG;
  if (n_new == 0) return IDX_OK;
  if (!raw_keys || !k_norm_w || !block_keys) return IDX_ERR_INVALID_ARG;
  if (!aligned(raw_keys, 2) || !aligned(k_norm_w, 4) || !aligned(block_keys, 4))
    return IDX_ERR_INVALID_ARG;
  return launch_block_pool(raw_keys, k_norm_w, block_keys, first_block, n_new, ratio, hd, rot, theta,
                           eps, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? IDX_OK
             : IDX_ERR_CUDA;
}

idx_status_t idx_qsa_qprep(const uint16_t *qk, const float *q_norm_w, float *q_out, uint32_t rows,
                           uint32_t first_pos, uint32_t qkw, uint32_t n_heads, uint32_t hd, uint32_t rot,
                           float theta, float eps, idx_stream_t stream) {
  if (hd < 32 || hd > 1024 || hd % 32 != 0 || rot % 2 != 0 || rot > hd) return IDX_ERR_INVALID_ARG;
  if (rows == 0 || n_heads == 0) return IDX_OK;
  if (static_cast<unsigned long long>(qkw) < static_cast<unsigned long long>(n_heads) * hd) return IDX_ERR_INVALID_ARG;
  if (rows > 0x7FFFFFFFu || n_heads > 65535u) return IDX_ERR_UNSUPPORTED;
  if (!qk || !q_norm_w || !q_out) return IDX_ERR_INVALID_ARG;
  if (!aligned(qk, 2) || !aligned(q_norm_w, 4) || !aligned(q_out, 4)) return IDX_ERR_INVALID_ARG;
  return launch_qsa_qprep(qk, q_norm_w, q_out, rows, first_pos, qkw, n_heads, hd, rot, theta, eps,
                          reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? IDX_OK
             : IDX_ERR_CUDA;
}

idx_status_t idx_expand_blocks(const int32_t *blocks, int32_t T, int32_t n_blocks, int32_t ratio,
                               int32_t *positions, idx_stream_t stream) {
  if (T < 0 || n_blocks < 0 || n_blocks > kMaxTopK || ratio < 1) return IDX_ERR_INVALID_ARG;
  if (T == 0 || n_blocks == 0) return IDX_OK;
  if (!blocks || !positions || !aligned(blocks, 4) || !aligned(positions, 4)) return IDX_ERR_INVALID_ARG;
  if (static_cast<long long>(n_blocks) * ratio > 0x7FFFFFFFLL) return IDX_ERR_INVALID_ARG;
  return launch_expand_blocks(blocks, T, n_blocks, ratio, positions,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? IDX_OK
             : IDX_ERR_CUDA;
}

idx_status_t idx_valid_lens_from_blocks(const int32_t *block_lens, int32_t T, int32_t epb,
                                        int32_t *valid_lens, idx_stream_t stream) {
  if (T < 0 || epb < 1) return IDX_ERR_INVALID_ARG;
  if (T == 0) return IDX_OK;
  if (!block_lens || !valid_lens || !aligned(block_lens, 4) || !aligned(valid_lens, 4))
    return IDX_ERR_INVALID_ARG;
  return launch_valid_lens(block_lens, T, epb, valid_lens, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? IDX_OK
             : IDX_ERR_CUDA;
}

const char *idx_status_string(idx_status_t status) {
  switch (status) {
    case IDX_OK: return "IDX_OK";
    case IDX_ERR_INVALID_ARG: return "IDX_ERR_INVALID_ARG";
    case IDX_ERR_UNSUPPORTED: return "IDX_ERR_UNSUPPORTED";
    case IDX_ERR_WORKSPACE_TOO_SMALL: return "IDX_ERR_WORKSPACE_TOO_SMALL";
    case IDX_ERR_CUDA: return "IDX_ERR_CUDA";
  }
  return "IDX_UNKNOWN_STATUS";
}

uint32_t idx_version(void) { return (1u << 16) | 0u; }

}  // extern "C"
