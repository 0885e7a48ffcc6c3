/*
 * idx.h — C ABI of libidx: the sparse-attention lightning indexer over a paged
 * NVFP4 key pool, QSA-style key pooling, and the selected-row K/V gather, for
 * one NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked "device" are CUDA device (or managed) memory owned by the
 *   caller; the library never frees or retains them and allocates nothing.
 * - Every call is asynchronous on `stream` (NULL = the legacy default stream).
 *   Nothing synchronises the host.
 * - The return value reports what the host can check before launching:
 *   IDX_ERR_INVALID_ARG (a null pointer, a negative size, a misaligned
 *   pointer), IDX_ERR_UNSUPPORTED (a legal shape this build has no kernel
 *   for), IDX_ERR_WORKSPACE_TOO_SMALL, IDX_ERR_CUDA (a launch error). On any
 *   error nothing has been launched.
 * - Bad data that only the device can see never faults and never traps: it
 *   ORs a bit into the optional device word `dev_status` (IDX_STATUS_*) and
 *   the affected outputs take their "empty" value (index -1, score -inf, a
 *   zero row). `dev_status` is never cleared by the library.
 * - `idx_stream_t` is the same handle as `cudaStream_t`.
 */
#ifndef IDX_H_
#define IDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *idx_stream_t;

typedef enum {
  IDX_OK = 0,
  IDX_ERR_INVALID_ARG = 1,
  IDX_ERR_UNSUPPORTED = 2,
  IDX_ERR_WORKSPACE_TOO_SMALL = 3,
  IDX_ERR_CUDA = 4
} idx_status_t;

/* Bits ORed into the caller's device status word. */
#define IDX_STATUS_BAD_BLOCK 1 /* a block-table entry outside [0, P)                       */
#define IDX_STATUS_BAD_LEN 2   /* a valid length outside [0, max_logical_blocks * epb]      */
#define IDX_STATUS_BAD_SEL 4   /* a gather position whose logical block is past the table   */
#define IDX_STATUS_TIMEOUT 8   /* an internal pipeline wait gave up (2 s); outputs invalid   */
#define IDX_STATUS_DEBUG_BOUNDS 16 /* debug-bounds builds only (-DIDX_DEBUG_BOUNDS): an index
                                      check failed and the access it guards was skipped    */

typedef enum { IDX_KEYS_NVFP4 = 0, IDX_KEYS_F32 = 1 } idx_key_format_t;

/* Which kernels idx_score_topk runs. AUTO picks the tensor-core path for
 * NVFP4 keys and the CUDA-core path for F32 keys. */
typedef enum { IDX_PATH_AUTO = 0, IDX_PATH_TENSOR = 1, IDX_PATH_SIMT = 2 } idx_path_t;

/* How the queries enter the dot products. EXACT: q as given (float32; the
 * tensor path is exact for q whose values are bf16). NVFP4 (opt-in, the
 * FP4-MMA phase that the header comment of "indexer_score_topk.cu" plans):
 * each head row of q is first quantised to NVFP4 exactly as
 * idx_quantize_q_nvfp4 states, and the scores are those of the quantised
 * queries, I[t,s] = sum_h w[t,h] * max(q_hat[t,h,:] . K[s,:], 0); the
 * tensor cores then take keys and queries in FP4 directly (block-scaled MMA),
 * with no decode of the keys. Tensor path and NVFP4 keys only, H <= 128. */
typedef enum { IDX_Q_EXACT = 0, IDX_Q_NVFP4 = 1 } idx_q_format_t;

/* Element type of q: float32, or bf16 bit patterns (the indexer projection's
 * output type; read as the exactly equal float32 values, so the results are
 * those of the upcast q). BF16 needs the tensor path. */
typedef enum { IDX_Q_F32 = 0, IDX_Q_BF16 = 1 } idx_q_dtype_t;

/*
 * idx_score_topk — lightning-indexer scores and their top-k.
 *
 * Computes, for every query t and every valid key s < valid_lens[t],
 *     I[t,s] = sum_h w[t,h] * max(q[t,h,:] . K[s,:], 0)
 * (eq. 16 in the header comment of "indexer_score_topk.cu",
 * nvfp4-megamoe-kernel dsv4/kernels/indexer; one key row per s shared by all
 * heads, as that page's main loop reads it), and returns TopK(I[t,:], top_k)
 * sorted by score descending, lower index first on equal scores, padded with
 * index -1 / score -inf when fewer than top_k keys are valid (the top-k
 * write-out section of the same page). -0.0 scores are reported as +0.0.
 *
 * Keys (the "Main kernel" argument list of that page):
 *   NVFP4: K[s,d] = e2m1(code) * e4m3(key_scale[row, d/16]) * key_gscale[phys]
 *     keys_fp4   device [P, epb, D/2] uint8, low nibble = even element d;
 *                E2M1 magnitudes {0,.5,1,1.5,2,3,4,6}, bit 3 the sign
 *                (commits 79ef87f and e74c844 of the indexer commit graph)
 *     key_scale  device [P, epb, D/16] uint8, FP8 E4M3 (OCP e4m3fn)
 *     key_gscale device [P] float32
 *   F32: keys_f32 device [P, epb, D] float32 (the QSA pooled keys of
 *     "metrale_model_layers/layers/ops/qsa.rs", qsa_score).
 * Slot resolution: lb = s / epb, slot = s % epb,
 *   phys = block_table[t * bt_stride + lb], row = phys * epb + slot.
 *   bt_stride = 0 makes every query read table row 0 (one sequence, many rows).
 *
 * Arguments (all sizes in elements):
 *   T >= 0, H in [1, 256], D: 128 (NVFP4) or 64/128 (F32)
 *   q          device [T, H, D], float32 or bf16 (q_dtype); the score_topk
 *              launcher of commit c2f705a upcasts bf16 to float32 first, a
 *              bf16 q here is read as those same float32 values
 *   w          device [T, H] float32
 *   P >= 1, entries_per_block (epb) >= 1; NVFP4 needs epb % 16 == 0
 *   block_table device int32, row t at block_table + t * bt_stride, with
 *              max_logical_blocks entries
 *   valid_lens device [T] int32
 *   top_k in [1, 4096]
 *   topk_idx   device [T, top_k] int32   (output)
 *   topk_score device [T, top_k] float32 (output)
 *   scores_out optional device [T, ld_scores] float32: when non-NULL, every
 *              I[t,s] (s < valid_lens[t]) is also written, -inf for keys of
 *              an out-of-range block; ld_scores >= max_logical_blocks * epb
 *   dev_status optional device int32 (IDX_STATUS_* bits ORed in)
 *   workspace  device scratch of at least idx_score_topk_workspace_size()
 *              bytes, 256-byte aligned. It needs no initialisation: every
 *              call writes each scratch word before it reads it (the q
 *              preparation kernel zeroes the key histograms and the
 *              selection's candidate counters). Calls that share a
 *              workspace must not overlap in time.
 *   path       idx_path_t
 *   num_ctas   CTAs of the persistent score kernel; 0 = one per SM
 *   timing_events optional pair of cudaEvent_t (as void*): when both are
 *              non-NULL, [0] is recorded on `stream` just before the q
 *              preparation and scoring kernels and [1] just after them (the
 *              selection kernel follows), so a caller can time the scoring
 *              alone. The second record keeps the selection kernel from
 *              launching early under the scorer's tail, which lengthens
 *              that call by a few microseconds.
 *   q_format   idx_q_format_t (0, the zero-initialised default, is EXACT).
 *   q_dtype    idx_q_dtype_t (0, the default, is F32); BF16 with the
 *              CUDA-core path gives IDX_ERR_UNSUPPORTED.
 *              NVFP4 with F32 keys, the CUDA-core path or H > 128 gives
 *              IDX_ERR_UNSUPPORTED; in that mode the key scale bytes are
 *              read as unsigned E4M3 (their sign bit must be clear).
 * Device-side errors: a table entry outside [0,P) drops that block's keys
 * (IDX_STATUS_BAD_BLOCK); a valid length outside [0, max_logical_blocks*epb]
 * pads that query's whole output (IDX_STATUS_BAD_LEN).
 */
typedef struct {
  int32_t T, H, D;
  const void *q;    /* float32 or bf16, per q_dtype */
  const float *w;
  int32_t key_format; /* idx_key_format_t */
  const uint8_t *keys_fp4;
  const uint8_t *key_scale;
  const float *key_gscale;
  const float *keys_f32;
  int32_t P, entries_per_block;
  const int32_t *block_table;
  int32_t max_logical_blocks;
  int64_t bt_stride;
  const int32_t *valid_lens;
  int32_t top_k;
  int32_t *topk_idx;
  float *topk_score;
  float *scores_out;
  int64_t ld_scores;
  int32_t *dev_status;
  void *workspace;
  size_t workspace_bytes;
  int32_t path;     /* idx_path_t */
  int32_t num_ctas; /* 0 = one per SM of the current device */
  void *timing_events[2];
  int32_t q_format; /* idx_q_format_t */
  int32_t q_dtype;  /* idx_q_dtype_t */
} idx_score_topk_args;

/* Bytes of workspace idx_score_topk needs for these arguments (host only; no
 * device work; with num_ctas == 0 it queries the current device's SM count).
 * Writes *bytes; returns IDX_ERR_INVALID_ARG / IDX_ERR_UNSUPPORTED like
 * idx_score_topk would. */
idx_status_t idx_score_topk_workspace_size(const idx_score_topk_args *args, size_t *bytes);

idx_status_t idx_score_topk(const idx_score_topk_args *args, idx_stream_t stream);

/*
 * idx_score_topk_static — idx_score_topk for callers that cannot allocate.
 *
 * The pages have no counterpart to this call; it exists for callers that may
 * not call cudaMalloc (for example an operator plugged into a host runtime
 * that owns all device memory and offers no allocator, or a serving loop that
 * must not allocate after start-up). It computes exactly what idx_score_topk
 * computes, with the same arguments, but ignores `workspace` and
 * `workspace_bytes`: its scratch is an array of IDX_STATIC_SCRATCH_BYTES
 * bytes inside the library's own device image, which every GPU that loads
 * libidx holds until the process exits. It calls no allocator.
 *   - Returns IDX_ERR_WORKSPACE_TOO_SMALL, without launching, when the
 *     arguments need more scratch than IDX_STATIC_SCRATCH_BYTES
 *     (idx_score_topk_workspace_size tells how much they need).
 *   - The first call on each device (with that device current) looks up the
 *     array's device address once; make that first call before any stream
 *     capture.
 *   - All calls share the one array: calls whose execution overlaps on the
 *     GPU race. Nothing in the array needs to start at zero.
 */
#define IDX_STATIC_SCRATCH_BYTES (8u << 20)
idx_status_t idx_score_topk_static(const idx_score_topk_args *args, idx_stream_t stream);

/*
 * idx_quantize_q_nvfp4 — the query quantisation of the NVFP4 q_format.
 *
 * The NVFP4 scheme of the keys ("FP4 dequantization (NVFP4 scheme)" section of
 * "indexer_score_topk.cu": E2M1 elements, one FP8 E4M3 scale per 16 elements)
 * plus one float32 scale per row that maps the row's largest |x| onto
 * 6 * 448 = 2688. For each row x of 128 values, with every operation one
 * float32 operation rounded to nearest:
 *     amax = max |x|;     gq = amax / 2688             (0 when amax == 0)
 *     group g of 16:      s_g = E4M3(ag / (6 * gq))    (ag: the group's max |x|)
 *     element d:          c_d = E2M1(x_d / (gq * s_g)), 0 when s_g == 0
 * E4M3() and E2M1() round to the nearest representable value, ties to the
 * even code, saturating at 448 and 6; a value rounding to zero gets code 0.
 * The row dequantises to gq * s_g * e2m1(c_d). q finite; rows whose largest
 * |x| is below 1e-30 are outside the contract (gq * s_g may underflow).
 *   q       device [rows, 128] float32, 16-byte aligned
 *   codes   device [rows, 64] uint8 (output): element 2j in the low nibble of
 *           byte j, E2M1 magnitude bits 0-2, sign bit 3
 *   scales  device [rows, 8] uint8 (output), E4M3
 *   gscale  device [rows] float32 (output)
 * Returns IDX_ERR_INVALID_ARG for rows < 0, a null or misaligned pointer.
 */
idx_status_t idx_quantize_q_nvfp4(const float *q, int64_t rows, uint8_t *codes, uint8_t *scales, float *gscale,
                                  idx_stream_t stream);

/*
 * idx_gather_kv — copy selected rows of a paged K/V cache into a dense tile.
 *
 * "metrale_model_layers/layers/ops/qsa.rs", qsa_gather: slot i of the output
 * holds position sel[t,i]; and the gather of commit c2f705a (indexer commit
 * graph): rows resolved through the block table. For p = sel[t,i] >= 0:
 *   phys = block_table[t * bt_stride + p / block_size], row p % block_size,
 *   k_out[t,i,:] = k_cache[phys, row, :] (bytes, unchanged), same for v.
 * p < 0 gives a zero row. p / block_size >= max_logical_blocks gives a zero
 * row and IDX_STATUS_BAD_SEL; phys outside [0,P) a zero row and
 * IDX_STATUS_BAD_BLOCK.
 *   sel          device [T, n_sel] int32
 *   k_cache, v_cache device [P, block_size, row_bytes] (any element type);
 *                v_cache / v_out may both be NULL (K only)
 *   row_bytes    > 0, multiple of 16; all four data pointers 16-byte aligned
 *   k_out, v_out device [T, n_sel, row_bytes]
 */
typedef struct {
  int32_t T, n_sel;
  const int32_t *sel;
  const int32_t *block_table;
  int32_t max_logical_blocks;
  int64_t bt_stride;
  int32_t P, block_size;
  const void *k_cache;
  const void *v_cache;
  int64_t row_bytes;
  void *k_out;
  void *v_out;
  int32_t *dev_status;
} idx_gather_kv_args;

idx_status_t idx_gather_kv(const idx_gather_kv_args *args, idx_stream_t stream);

/*
 * idx_gather_split — the dense BF16 tile of selected positions from a paged
 * cache whose rows are split into an FP8 part and a BF16 part.
 *
 * "Commit graph, dsv4/kernels/indexer", commit c2f705a (gather_kv.cu): one
 * output row per (query, top-k entry), rows resolved through the block
 * table, FP8 dequantised to BF16, the BF16 part copied. The commit gives no
 * layout; this one: for p = sel[t,i] resolved to (phys, row) exactly as in
 * idx_gather_kv, with s = nope_scale ? nope_scale[phys, row] : 1,
 *   out[t,i, d]            = bf16_rn(float(e4m3(nope[phys,row,d])) * s), d < nope_dim
 *   out[t,i, nope_dim + d] = rope[phys,row,d],                           d < rope_dim
 * (float multiply, then round to nearest even). p < 0 gives a zero row;
 * a logical block past max_logical_blocks a zero row and IDX_STATUS_BAD_SEL;
 * phys outside [0,P) a zero row and IDX_STATUS_BAD_BLOCK.
 *   sel          device [T, n_sel] int32
 *   nope         device [P, block_size, nope_dim] FP8 E4M3 (OCP e4m3fn)
 *   nope_scale   device [P, block_size] float32, or NULL
 *   rope         device [P, block_size, rope_dim] bf16 (raw bit patterns)
 *   out          device [T, n_sel, nope_dim + rope_dim] bf16
 *   nope_dim a multiple of 4, rope_dim even; pointers 4-byte aligned
 */
typedef struct {
  int32_t T, n_sel;
  const int32_t *sel;
  const int32_t *block_table;
  int32_t max_logical_blocks;
  int64_t bt_stride;
  int32_t P, block_size;
  const uint8_t *nope;
  const float *nope_scale;
  const uint16_t *rope;
  int32_t nope_dim, rope_dim;
  uint16_t *out;
  int32_t *dev_status;
} idx_gather_split_args;

idx_status_t idx_gather_split(const idx_gather_split_args *args, idx_stream_t stream);

/*
 * idx_block_pool — pool newly complete blocks of raw keys into block keys.
 *
 * "metrale_model_layers/layers/ops/qsa.rs", qsa_block_pool: for block
 * b = first_block + i, i < n_new: the mean m of raw rows
 * [b*ratio, (b+1)*ratio), then y = m / sqrt(mean(m^2) + eps) * (1 + w), then
 * rope on the first `rot` dimensions at position b*ratio, pairing d with
 * d + rot/2 at angle pos * theta^(-2d/rot) (d < rot/2). The angle is formed
 * and reduced to [-pi, pi] in double precision; its sine and cosine are
 * taken in single precision.
 *   raw_keys    device [(first_block+n_new)*ratio, hd] bf16 (raw bit patterns)
 *   k_norm_w    device [hd] float32
 *   block_keys  device [first_block + n_new, hd] float32; rows
 *               first_block .. first_block+n_new-1 are written
 *   hd a multiple of 32 in [32, 1024]; rot even, rot <= hd; ratio >= 1
 * n_new == 0 returns IDX_OK without launching (as qsa_block_pool does).
 */
idx_status_t idx_block_pool(const uint16_t *raw_keys, const float *k_norm_w, float *block_keys,
                            uint32_t first_block, uint32_t n_new, uint32_t ratio, uint32_t hd,
                            uint32_t rot, float theta, float eps, idx_stream_t stream);

/*
 * idx_qsa_qprep — query preparation for QSA block scoring.
 *
 * "metrale_model_layers/layers/ops/qsa.rs", qsa_qprep (one decode query) and
 * qsa_qprep_rows (prefill rows): for row r < rows and head h < n_heads, the
 * head's q x = qk[r*qkw + h*hd .. + hd), then y = x / sqrt(mean(x^2) + eps) *
 * (1 + w), then rope on the first `rot` dimensions at position first_pos + r,
 * pairing d with d + rot/2 exactly as idx_block_pool does.
 *   qk        device [rows, qkw] bf16 (raw bit patterns): rows of the indexer
 *             projection; head h's q at columns h*hd .. h*hd+hd-1
 *   q_norm_w  device [hd] float32
 *   q_out     device [rows, n_heads, hd] float32
 *   hd a multiple of 32 in [32, 1024]; rot even, rot <= hd; qkw >= n_heads*hd
 * A decode query is rows = 1, first_pos = its position, qkw = n_heads*hd.
 * rows == 0 or n_heads == 0 returns IDX_OK without launching.
 */
idx_status_t idx_qsa_qprep(const uint16_t *qk, const float *q_norm_w, float *q_out, uint32_t rows,
                           uint32_t first_pos, uint32_t qkw, uint32_t n_heads, uint32_t hd, uint32_t rot,
                           float theta, float eps, idx_stream_t stream);

/*
 * idx_qsa_prefill_attn — prefill attention over the selected blocks plus the
 * incomplete tail.
 *
 * "metrale_model_layers/layers/ops/qsa.rs", qsa_prefill_attn: row r sits at
 * position p = first_pos + r; blocks of `ratio` tokens b < (p+1)/ratio are
 * complete. For each row and query head h, one softmax over
 * (q[r,h] . K[t]) * inv_sqrt_d for every token t of each selected block
 * b = lists[r*topk + i] with 0 <= b < (p+1)/ratio (other entries are
 * skipped; duplicates count twice) and every tail token
 * ((p+1)/ratio)*ratio <= t <= p, with K and V of kv head h / (nq/nkv);
 * attn_out[r,h] = sum softmax * V. A row with no token gets zeros.
 *   q            device [rows, nq, hd] float32
 *   k_cache,
 *   v_cache      device [P, block_size, nkv, hd] bf16 (raw bit patterns);
 *                token t lives in page block_table[t / block_size], slot
 *                t % block_size
 *   block_table  device [n_pages] int32 (one sequence)
 *   lists        device [rows, topk] int32 block ids (NULL when topk == 0)
 *   attn_out     device [rows, nq, hd] float32
 *   hd in {64, 128, 256}; nq a multiple of nkv; ratio, block_size >= 1
 * Alignment: q, block_table, lists, attn_out 4 bytes; k_cache and v_cache
 * 8 bytes (IDX_ERR_INVALID_ARG otherwise). With 1, 2, 4 or 8 query heads per
 * kv head, hd <= 128 and both caches 16-byte aligned the tiled kernel runs;
 * otherwise the per-head kernel (same result up to rounding order).
 * Device-side errors: a token whose page index is past n_pages or whose page
 * is outside [0,P) is left out (IDX_STATUS_BAD_BLOCK in *dev_status).
 * rows == 0 or nq == 0 returns IDX_OK without launching.
 */
idx_status_t idx_qsa_prefill_attn(const float *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  const int32_t *block_table, int32_t n_pages, int32_t P, const int32_t *lists,
                                  float *attn_out, uint32_t rows, uint32_t first_pos, uint32_t topk,
                                  uint32_t ratio, uint32_t block_size, uint32_t nq, uint32_t nkv, uint32_t hd,
                                  float inv_sqrt_d, int32_t *dev_status, idx_stream_t stream);

/*
 * idx_expand_blocks — token positions of selected blocks, for idx_gather_kv.
 *
 * qsa.rs, qsa_gather fills slot i with position sel[i]; the page does not
 * say in which order blocks are laid out. This call takes the selected block
 * indices of each query (blocks [T, n_blocks], -1 = none, any order, e.g. a
 * top-k output), sorts them ascending and writes each block's `ratio`
 * positions b*ratio .. b*ratio+ratio-1 in order, then -1 in the unused tail:
 *   positions device [T, n_blocks * ratio] int32.
 * n_blocks in [0, 4096], ratio >= 1.
 */
idx_status_t idx_expand_blocks(const int32_t *blocks, int32_t T, int32_t n_blocks, int32_t ratio,
                               int32_t *positions, idx_stream_t stream);

/*
 * idx_valid_lens_from_blocks — valid_lens[t] = block_lens[t] * epb.
 * compute_valid_lens of commit c2f705a (every entry of an allocated block is
 * valid).  block_lens, valid_lens: device [T] int32.
 */
idx_status_t idx_valid_lens_from_blocks(const int32_t *block_lens, int32_t T, int32_t epb,
                                        int32_t *valid_lens, idx_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *idx_status_string(idx_status_t status);

/* Library ABI version, (major << 16) | minor. */
uint32_t idx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H_ */
