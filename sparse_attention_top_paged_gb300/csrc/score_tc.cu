// score_tc.cu — tensor-core (tcgen05) lightning-indexer scorer.
//
// What it computes: eq. 16 of "indexer_score_topk.cu" (nvfp4-megamoe-kernel,
// dsv4/kernels/indexer), I[t,s] = sum_h w[t,h] * ReLU(q[t,h] . K[s]), over NVFP4
// keys resolved through the block table, written to a [T, ld] score matrix;
// the selection kernels in topk.cu then take TopK(I[t,:], k).
// That page's kernel runs one CTA per query with scalar FP32 dot products and
// a locked shared heap; here two kernels run back to back (the second may
// start before the first ends):
//
// qprep_kernel turns q into the MMA's B operand once, as records in global
// memory. A record serves a "row group" of R query rows: R = 2 when every row
// reads the same block table (one sequence, many rows), so one decoded key
// tile feeds both rows' dot products in a single MMA of N = 2 Npad; else R = 1.
// Per head row: a power-of-two scale 2^sigma, f16 hi and lo parts (the lo
// part only feeds the MMA when some q value is not exact in f16, e.g.
// bf16-valued q never needs it), w' = w 2^-sigma and the lo flags. It also
// zeroes the per-query key histograms (and the selection's candidate
// counters), so the workspace needs no initialisation.
//
// score_tc_kernel is a persistent, warp-specialised pipeline:
//   work     The tiles of 128 consecutive keys of every row group, laid end to
//            end, are split evenly over the CTAs (one per SM). A "segment" is
//            a CTA's run of tiles of one row group (it shares one B operand).
//   warp 18  resolver: looks up block-table entries and per-block global
//            scales 32 blocks at a time (one per lane) into a ring of per-tile
//            records, so no dependent global load sits on the copy path.
//   warp 0   producer: streams each tile's packed E2M1 nibbles (2-D TMA,
//            64-byte swizzle) and E4M3 scales (1-D bulk copy) into a ring of
//            shared-memory stages, several tiles at once (one per lane), and
//            at each segment start copies the query's q record into one of
//            two segment slots.
//   warps 2-5 decoders: one thread per key row decodes 128 elements
//            e2m1 * e4m3 exactly into f16 (hardware converts) and stores them
//            to tensor memory as the MMA's A operand.
//   warp 1   MMA issuer: D[128 keys x R Npad heads] = A * B^T in f32, K = 128, as
//            8 (or 16 with the lo part) tcgen05.mma kind::f16 steps.
//   warps 6-17 epilogue, three groups of four taking tiles in turn: one
//            thread per key reads its accumulator row (32 columns at a
//            time) from tensor memory and forms, per row of the group,
//            I = g * sum_h (w_h 2^-sigma_h) relu(acc_h)
//            (the per-block global scale g is factored out, so relu(g a) = g
//            relu(a) for g > 0 and g min(a,0) for g < 0), then stores I to the
//            score matrix (coalesced: a warp writes 32 consecutive keys). The
//            epilogue warps never wait for one another.
//
// Products e2m1 * e4m3 are exact in f16, and bf16-valued q is exact in the
// scaled f16 hi part, so a single MMA pass computes the dot products with f32
// accumulation only; full-precision f32 q takes the second (lo) pass.
//
// NVFP4-q mode (opt-in, the FP4-MMA phase that page's header comment plans):
// qprep quantises each head of q to NVFP4 (nvfp4q.cuh) and the MMA is
// tcgen05.mma kind::mxf4nvf4, which reads the keys' packed E2M1 nibbles
// straight from the TMA stage and the q codes from the record, with the E4M3
// group scales of both from tensor memory: nothing is decoded. The decoder
// warps only copy each tile's key scales and the segment's q scales into the
// tile's tensor-memory scale slot; the per-head float32 scale gq is folded
// into w' (relu(gq a) = gq relu(a), gq >= 0). The stage is handed back when
// the tile's MMAs complete.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "nvfp4q.cuh"
#include "tc_ptx.cuh"

namespace idx {
namespace {

constexpr int kDecWarps = 4;                       // 4: a warp decodes whole rows; 8: half rows
constexpr int kEpiGroups = 3;                      // epilogue groups of four warps
constexpr int kEpiWarp0 = 2 + kDecWarps;           // first epilogue warp
constexpr int kResolverWarp = kEpiWarp0 + 4 * kEpiGroups;   // after the epilogue warps
constexpr int kThreads = 32 * (kResolverWarp + 1);
constexpr int kTileKeys = 128;
constexpr int kMaxNS = 16;               // raw stages (as many as shared memory holds)
constexpr int kR = 64;                   // metadata ring (tiles)
constexpr uint32_t kStageBytes = 9216;   // 128 x 64 B nibbles + 128 x 8 B scales
constexpr uint32_t kScaleOff = 8192;
constexpr int kMaxBlocksPerTile = 8;     // epb >= 16
// A pipeline wait gives up after kTimeoutNs, raising the CTA's abort flag
// (IDX_STATUS_TIMEOUT); the waits that drain asynchronous work before exit
// always allow kDrainNs. Builds for the failure-path test shorten the first
// (IDX_WAIT_LIMIT_NS).
#ifdef IDX_WAIT_LIMIT_NS
constexpr uint64_t kTimeoutNs = IDX_WAIT_LIMIT_NS;
#else
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
#endif
constexpr uint64_t kDrainNs = 2000000000ull;
constexpr int kSmemLimit = 227 * 1024;

// One tile's resolved blocks, written by the resolver warp, read by the
// producer (physical blocks) and the epilogue (global scales, validity).
struct MetaEntry {
  int phys[kMaxBlocksPerTile];
  float g[kMaxBlocksPerTile];
  uint32_t mask;  // bit b: block b of the tile resolved to a valid physical block
  int lb0;        // first logical block of the tile
  int s0;         // first key of the tile
  int nblk;       // blocks the tile touches (up to its last valid key)
  int t;          // the tile's row group
  int seg;        // first tile of the CTA's segment number seg - 1; 0: not a segment start
  int len[2];     // keys of each row of the group (0: no such row, or a bad length)
  int pad_[8];
};
static_assert(sizeof(MetaEntry) == 128, "meta entry");

// Per-row-group B-operand record, written by qprep_kernel to global memory and
// copied verbatim into a shared-memory segment slot: f16 hi rows, f16 lo rows
// (each NR = R Npad head rows x 128 dims, K-major, 128-byte swizzled), w' (NR
// floats), lo flags (NR ints). Head row n holds head n % Npad of row
// R * group + n / Npad.
// NVFP4-q records instead hold the E2M1 codes (NR rows x 64 bytes, K-major,
// 64-byte swizzled), then the E4M3 group scales as 1 KB of 32-bit words laid
// out for the tensor-memory scale slot (word (c * 4 + j) * 32 + l: the four
// scales of K step c of head row l + 32 j; zero past NR), then w' = w gq.
struct TcLayout {
  int Npad, R, NR, nq, nseg, na, nd, ne, ns, box_rows, bpt, epb_shift;
  int fp4;          // NVFP4-q mode
  uint32_t a_cols;  // tensor-memory columns per A slot (decoded keys; or the scale slot)
  uint32_t b_bytes, sfb_off, rec_w, rec_flags, rec_bytes, rec_smem;
  uint32_t off_b, off_raw, off_meta, off_bar, off_misc;
  uint32_t smem_bytes;
};

// barrier indices (uint64 slots from off_bar)
constexpr int kMaxSlots = 4;  // tensor-memory A and D slots (each)
constexpr int B_FULL_RAW = 0, B_EMPTY_RAW = kMaxNS, B_FULL_A = 2 * kMaxNS, B_EMPTY_A = B_FULL_A + kMaxSlots,
              B_FULL_D = B_EMPTY_A + kMaxSlots, B_EMPTY_D = B_FULL_D + kMaxSlots,
              B_META_FULL = B_EMPTY_D + kMaxSlots, B_META_EMPTY = B_META_FULL + kR, B_SEG_FULL = B_META_EMPTY + kR,
              B_SEG_BFREE = B_SEG_FULL + 2, B_SEG_WFREE = B_SEG_FULL + 4, B_DRAIN = B_SEG_FULL + 6,
              B_NEVER = B_DRAIN + 1, B_COUNT = B_NEVER + 1;

// misc ints
constexpr int M_TMEM = 0, M_ABORT = 1, M_T0 = 2, M_J0 = 3, M_SCAN = 8;  // then one long per warp (scan)
constexpr uint32_t kMiscBytes = 8 * 4 + (kThreads / 32) * 8;

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Keys of row t, or 0 for a length outside [0, max_lb * epb] (such a row is
// padded by the selection and reported there).
__device__ __forceinline__ int row_len(const ScoreParams &p, int t) {
  const int L = p.valid_lens[t];
  return (L <= 0 || static_cast<long long>(L) > static_cast<long long>(p.max_lb) * p.epb) ? 0 : L;
}

// Tiles of row group tq (kRows rows): its longest valid row, in 128-key tiles.
template <int kRows>
__device__ __forceinline__ int ntiles_of(const ScoreParams &p, int tq) {
  int L = row_len(p, tq * kRows);
  if (kRows > 1 && tq * kRows + 1 < p.T) L = max(L, row_len(p, tq * kRows + 1));
  return (L + kTileKeys - 1) / kTileKeys;
}

// Deterministic walk over a CTA's tiles; every role runs its own copy.
template <int kRows>
struct Walker {
  int t, j, nt;   // row group, tile within it, its tile count
  __device__ void init(const ScoreParams &p, const TcLayout &lay, int t0, int j0) {
    t = t0;
    j = j0;
    nt = (t0 < lay.nq) ? ntiles_of<kRows>(p, t0) : 0;
  }
  __device__ void next(const ScoreParams &p, const TcLayout &lay) {
    if (++j == nt) {
      j = 0;
      do {
        ++t;
      } while (t < lay.nq && (nt = ntiles_of<kRows>(p, t)) == 0);
    }
  }
};

// Slot and phase parity of a ring of mbarrier-guarded buffers, advanced one use
// at a time (no division in the per-tile loops). Consumers wait on "full" with
// `phase`; producers wait on "empty" with `phase ^ 1` (a fresh barrier counts
// as having completed that phase).
struct Ring {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Block-wide inclusive scan of one long long per thread (all kThreads threads).
__device__ long long block_incl_scan(long long v, long long *scratch, long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const long long s = scratch[w];
    if (w < warp) before += s;
    all += s;
  }
  __syncthreads();
  *total = all;
  return before + x;
}

// q -> the B-operand record of row group tq: one block per record, one warp
// per head row at a time, 4 dims per lane (head rows of absent rows or heads
// are zero). load_head_row reads this lane's part of head row n.
// Exact q: per head a power-of-two scale 2^sigma puts the largest |q| in
// [2^14, 2^15) (sigma from the exponent field; subnormal or zero heads keep
// sigma 0; clamped so 2^sigma and 2^-sigma are normal floats); the scaled
// values are split into f16 hi + lo and w' = w 2^-sigma undoes the scale
// after the ReLU. The lo part is written only when some head of the record
// has a non-zero lo (never for bf16-valued q short of a 2^-31 dynamic range
// within a head): the MMA reads it only then (the OR of the heads' flags).
// NVFP4 q: the quantisation of nvfp4q.cuh, w' = w gq.
// The raw loads (a float4, or four bf16 in .x/.y) are kept apart from their
// conversion (head_row_values) so several rows' loads can be in flight.
__device__ __forceinline__ void load_head_row(const ScoreParams &p, const TcLayout &lay, int tq, int n, int lane,
                                              uint4 &raw, float &wv) {
  const int h = n % lay.Npad, t = tq * lay.R + n / lay.Npad;
  raw = make_uint4(0u, 0u, 0u, 0u);
  wv = 0.0f;
  if (h < p.H && t < p.T) {
    const long long e0 = (static_cast<long long>(t) * p.H + h) * 128;
    if (p.q16 != nullptr) {
      const uint2 u = reinterpret_cast<const uint2 *>(p.q16 + e0)[lane];
      raw.x = u.x;
      raw.y = u.y;
    } else {
      raw = reinterpret_cast<const uint4 *>(p.q + e0)[lane];
    }
    wv = p.w[static_cast<long long>(t) * p.H + h];
  }
}

// This lane's 4 values of a head row from its raw load (bf16: the float32
// with the same leading 16 bits).
__device__ __forceinline__ float4 head_row_values(const ScoreParams &p, uint4 raw) {
  if (p.q16 != nullptr)
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
  return make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z), __uint_as_float(raw.w));
}

// The exact-q split of this lane's 4 values of head row n: its offset in the
// hi (and lo) rows, the packed f16 hi and lo, and w'. Returns whether this
// warp's head row has a non-zero lo part.
__device__ __forceinline__ bool split_head_row(const TcLayout &lay, int n, int lane, float4 x, float wv, uint32_t &off,
                                               uint2 &vh, uint2 &vl, float &wq) {
  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  const int sigma = (ex == 0) ? 0 : max(-126, min(126, 141 - ex));
  const float up = __uint_as_float(static_cast<uint32_t>(127 + sigma) << 23);
  const float down = __uint_as_float(static_cast<uint32_t>(127 - sigma) << 23);
  const float xs[4] = {x.x * up, x.y * up, x.z * up, x.w * up};
  __half hi[4], lo[4];
  bool any_lo = false;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hi[e] = __float2half_rn(xs[e]);
    lo[e] = __float2half_rn(xs[e] - __half2float(hi[e]));
    any_lo |= (__half2float(lo[e]) != 0.0f);
  }
  // dims 4*lane .. 4*lane+3: K block kb = lane / 16 (64 dims each), 16-byte
  // chunk jj = (lane / 2) % 8 of the head row's 128 bytes, swizzled by n % 8
  const int ch = lane >> 1, kb = ch >> 3, jj = ch & 7;
  off = kb * (lay.NR * 128) + n * 128 + ((jj ^ (n & 7)) * 16) + (lane & 1) * 8;
  vh.x = static_cast<uint32_t>(__half_as_ushort(hi[0])) | (static_cast<uint32_t>(__half_as_ushort(hi[1])) << 16);
  vh.y = static_cast<uint32_t>(__half_as_ushort(hi[2])) | (static_cast<uint32_t>(__half_as_ushort(hi[3])) << 16);
  vl.x = static_cast<uint32_t>(__half_as_ushort(lo[0])) | (static_cast<uint32_t>(__half_as_ushort(lo[1])) << 16);
  vl.y = static_cast<uint32_t>(__half_as_ushort(lo[2])) | (static_cast<uint32_t>(__half_as_ushort(lo[3])) << 16);
  wq = wv * down;
  return __any_sync(0xFFFFFFFFu, any_lo);
}

// One block per record (many records: as many blocks as records fill the
// GPU); the lo rows only when needed.
__global__ void __launch_bounds__(256) qprep_kernel(ScoreParams p, TcLayout lay, uint8_t *__restrict__ rec,
                                                    uint32_t *__restrict__ hist, uint32_t *__restrict__ cand_cnt) {
  ptx::launch_dependents();  // the scorer may start its prologue meanwhile
  constexpr int kWarps = 8, kAhead = 4;
  const int tq = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the group's rows: zero their key histograms (and candidate counters)
  for (int rr = 0; rr < lay.R; ++rr) {
    const int t = tq * lay.R + rr;
    if (t >= p.T) break;
    uint4 *hz = reinterpret_cast<uint4 *>(hist + static_cast<size_t>(t) * kScoreBins);
    for (int i = threadIdx.x; i < kScoreBins / 4; i += blockDim.x) hz[i] = make_uint4(0u, 0u, 0u, 0u);
    if (cand_cnt != nullptr && threadIdx.x == 0) cand_cnt[t] = 0u;
  }
  uint8_t *r = rec + static_cast<size_t>(tq) * lay.rec_bytes;
  if (lay.fp4) {   // scale words of head rows NR .. 127 stay zero
    uint32_t *sw = reinterpret_cast<uint32_t *>(r + lay.sfb_off);
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
      if (((i >> 5) & 3) * 32 >= lay.NR) sw[i] = 0u;
  }
  bool any_lo = false;
  for (int nb = warp; nb < lay.NR; nb += kAhead * kWarps) {
    uint4 raw[kAhead];
    float wv[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int n = nb + u * kWarps;
      if (n < lay.NR) load_head_row(p, lay, tq, n, lane, raw[u], wv[u]);
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int n = nb + u * kWarps;
      if (n >= lay.NR) continue;
      const float4 xu = head_row_values(p, raw[u]);
      if (lay.fp4) {
        uint32_t codes16, scale;
        float gq;
        nvfp4_quantize_lane(xu, codes16, scale, gq);
        // codes: bytes 2 lane, 2 lane + 1 of head row n (64 bytes, 64-byte swizzle in 8-row groups)
        const uint32_t off =
            (n >> 3) * 512 + (n & 7) * 64 + ((((lane >> 3) ^ ((n >> 1) & 3)) & 3) * 16) + ((2 * lane) & 15);
        *reinterpret_cast<uint16_t *>(r + off) = static_cast<uint16_t>(codes16);
        if ((lane & 3) == 0) {   // scale of group g = lane / 4: K step g / 4, byte g % 4 of its word
          const int g = lane >> 2;
          r[lay.sfb_off + (((g >> 2) * 4 + (n >> 5)) * 32 + (n & 31)) * 4 + (g & 3)] = static_cast<uint8_t>(scale);
        }
        if (lane == 0) {
          reinterpret_cast<float *>(r + lay.rec_w)[n] = __fmul_rn(wv[u], gq);
          reinterpret_cast<int *>(r + lay.rec_flags)[n] = 0;
        }
      } else {
        uint32_t off;
        uint2 vh, vl;
        float wq;
        const bool row_lo = split_head_row(lay, n, lane, xu, wv[u], off, vh, vl, wq);
        *reinterpret_cast<uint2 *>(r + off) = vh;
        any_lo |= row_lo;
        if (lane == 0) {
          reinterpret_cast<float *>(r + lay.rec_w)[n] = wq;
          reinterpret_cast<int *>(r + lay.rec_flags)[n] = row_lo ? 1 : 0;
        }
      }
    }
  }
  // The lo rows, only when the MMA will read them: some head of the record
  // has a non-zero lo (then every head's lo, zeros included, is written).
  if (lay.fp4 || !__syncthreads_or(any_lo)) return;
  for (int n = warp; n < lay.NR; n += kWarps) {
    uint4 raw;
    float wv;
    load_head_row(p, lay, tq, n, lane, raw, wv);
    uint32_t off;
    uint2 vh, vl;
    float wq;
    split_head_row(lay, n, lane, head_row_values(p, raw), wv, off, vh, vl, wq);
    *reinterpret_cast<uint2 *>(r + lay.b_bytes + off) = vl;
  }
}

// Few records: block (tq, y) prepares head rows 8y .. 8y+7 of record tq, one
// warp each, so the work spreads over more blocks; every head's lo row is
// written (the blocks of a record cannot agree on skipping it).
__global__ void __launch_bounds__(256) qprep_rows_kernel(ScoreParams p, TcLayout lay, uint8_t *__restrict__ rec,
                                                         uint32_t *__restrict__ hist, uint32_t *__restrict__ cand_cnt) {
  ptx::launch_dependents();  // the scorer may start its prologue meanwhile
  const int tq = blockIdx.x;
  for (int rr = 0; rr < lay.R; ++rr) {
    // the blocks of the group zero its rows' key histograms between them
    // (and their candidate counters, when given)
    const int t = tq * lay.R + rr;
    if (t >= p.T) break;
    uint32_t *hz = hist + static_cast<size_t>(t) * kScoreBins;
    for (int i = blockIdx.y * blockDim.x + threadIdx.x; i < kScoreBins; i += gridDim.y * blockDim.x) hz[i] = 0u;
    if (cand_cnt != nullptr && blockIdx.y == 0 && threadIdx.x == 0) cand_cnt[t] = 0u;
  }
  const int n = blockIdx.y * 8 + static_cast<int>(threadIdx.x >> 5);   // head row of the record
  const int lane = threadIdx.x & 31;
  uint8_t *r = rec + static_cast<size_t>(tq) * lay.rec_bytes;
  if (lay.fp4 && blockIdx.y == 0) {   // scale words of head rows NR .. 127 stay zero
    uint32_t *sw = reinterpret_cast<uint32_t *>(r + lay.sfb_off);
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
      if (((i >> 5) & 3) * 32 >= lay.NR) sw[i] = 0u;
  }
  if (n >= lay.NR) return;
  uint4 raw;
  float wv;
  load_head_row(p, lay, tq, n, lane, raw, wv);
  const float4 x = head_row_values(p, raw);
  if (lay.fp4) {
    uint32_t codes16, scale;
    float gq;
    nvfp4_quantize_lane(x, codes16, scale, gq);
    const uint32_t off = (n >> 3) * 512 + (n & 7) * 64 + ((((lane >> 3) ^ ((n >> 1) & 3)) & 3) * 16) + ((2 * lane) & 15);
    *reinterpret_cast<uint16_t *>(r + off) = static_cast<uint16_t>(codes16);
    if ((lane & 3) == 0) {
      const int g = lane >> 2;
      r[lay.sfb_off + (((g >> 2) * 4 + (n >> 5)) * 32 + (n & 31)) * 4 + (g & 3)] = static_cast<uint8_t>(scale);
    }
    if (lane == 0) {
      reinterpret_cast<float *>(r + lay.rec_w)[n] = __fmul_rn(wv, gq);
      reinterpret_cast<int *>(r + lay.rec_flags)[n] = 0;
    }
    return;
  }
  uint32_t off;
  uint2 vh, vl;
  float wq;
  const bool row_lo = split_head_row(lay, n, lane, x, wv, off, vh, vl, wq);
  *reinterpret_cast<uint2 *>(r + off) = vh;
  *reinterpret_cast<uint2 *>(r + lay.b_bytes + off) = vl;
  if (lane == 0) {
    reinterpret_cast<float *>(r + lay.rec_w)[n] = wq;
    reinterpret_cast<int *>(r + lay.rec_flags)[n] = row_lo ? 1 : 0;
  }
}

template <int kRows, bool kFp4>
__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmap_nib, ScoreParams p, TcLayout lay,
                    const uint8_t *__restrict__ qrec, uint32_t *__restrict__ hist, float *__restrict__ scores,
                    long long ld) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array, so accesses through sm stay shared-space ones
  uint8_t *sm = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + lay.off_bar);
  int *misc = reinterpret_cast<int *>(sm + lay.off_misc);
  volatile int *abort_flag = misc + M_ABORT;
  auto bar = [&](int i) { return ptx::smem_addr(bars + i); };

  if (warp == 0) {   // the barriers, spread over the warp's lanes (the metadata ring alone has 2 kR)
    if (lane == 0) ptx::launch_dependents();  // the selection kernel may be scheduled as CTAs of this one finish
    for (int s = lane; s < lay.ns; s += 32) {
      ptx::mbar_init(bar(B_FULL_RAW + s), 1);
      ptx::mbar_init(bar(B_EMPTY_RAW + s), kFp4 ? 1 : kDecWarps);   // decoders, or the MMA commit
    }
    if (lane < kMaxSlots) {
      ptx::mbar_init(bar(B_FULL_A + lane), kDecWarps);
      ptx::mbar_init(bar(B_EMPTY_A + lane), 1);
      ptx::mbar_init(bar(B_FULL_D + lane), 1);
      ptx::mbar_init(bar(B_EMPTY_D + lane), 4);
    }
    if (lane < 2) {
      ptx::mbar_init(bar(B_SEG_FULL + lane), 1);   // producer (record copy)
      ptx::mbar_init(bar(B_SEG_BFREE + lane), 1);
      ptx::mbar_init(bar(B_SEG_WFREE + lane), 4 * kEpiGroups);  // one arrive per epilogue warp
    }
    for (int r = lane; r < kR; r += 32) {
      ptx::mbar_init(bar(B_META_FULL + r), 1);   // resolver
      ptx::mbar_init(bar(B_META_EMPTY + r), 4);  // epilogue warps
    }
    if (lane == 0) {
      ptx::mbar_init(bar(B_DRAIN), 1);   // MMA commit before exit
      ptx::mbar_init(bar(B_NEVER), 1);   // nothing arrives (failure-path test builds only)
      misc[M_ABORT] = 0;
    }
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(ptx::smem_addr(misc + M_TMEM), 512);

  // ---- work partition: tiles [g0, g1) of the concatenated tile list ----
  long long *scan = reinterpret_cast<long long *>(misc + M_SCAN);
  const long long G = gridDim.x, c = blockIdx.x;
  long long g0 = 0, g1 = 0;
  if (lay.nq <= kThreads) {
    // one row group per thread: a single scan gives the total and each group's range
    const long long v = (static_cast<int>(threadIdx.x) < lay.nq) ? ntiles_of<kRows>(p, threadIdx.x) : 0;
    long long total;
    const long long incl = block_incl_scan(v, scan, &total);
    const long long qg = total / G, rg = total % G;
    g0 = c * qg + (c * rg) / G;
    g1 = (c + 1) * qg + ((c + 1) * rg) / G;
    const long long excl = incl - v;
    if (v > 0 && excl <= g0 && g0 < incl) {   // exactly one thread when g0 < total
      misc[M_T0] = static_cast<int>(threadIdx.x);
      misc[M_J0] = static_cast<int>(g0 - excl);
    }
    if (threadIdx.x == 0 && g0 >= total) {
      misc[M_T0] = lay.nq;
      misc[M_J0] = 0;
    }
  } else {
    long long total = 0;
    {
      long long local = 0;
      for (int t = threadIdx.x; t < lay.nq; t += kThreads) local += ntiles_of<kRows>(p, t);
      long long tot;
      block_incl_scan(local, scan, &tot);
      total = tot;
    }
    const long long qg = total / G, rg = total % G;
    g0 = c * qg + (c * rg) / G;
    g1 = (c + 1) * qg + ((c + 1) * rg) / G;
    if (threadIdx.x == 0) {
      misc[M_T0] = lay.nq;
      misc[M_J0] = 0;
    }
    __syncthreads();
    long long base = 0;
    for (int chunk = 0; chunk < lay.nq; chunk += kThreads) {
      const int t = chunk + threadIdx.x;
      const long long v = (t < lay.nq) ? ntiles_of<kRows>(p, t) : 0;
      long long tot;
      const long long incl = block_incl_scan(v, scan, &tot);
      const long long excl = incl - v;
      if (v > 0 && base + excl <= g0 && g0 < base + incl) {
        misc[M_T0] = t;
        misc[M_J0] = static_cast<int>(g0 - (base + excl));
      }
      base += tot;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[M_TMEM]);
  const int t0 = misc[M_T0], j0 = misc[M_J0];
  const int n_tiles = (g0 < g1) ? static_cast<int>(g1 - g0) : 0;
  const int Npad = lay.Npad, NR = lay.NR, nseg = lay.nseg, na = lay.na, nd = lay.nd;
  const uint32_t b_bytes = lay.b_bytes;
  uint8_t *sB = sm + lay.off_b;
  uint8_t *sRaw = sm + lay.off_raw;
  MetaEntry *sMeta = reinterpret_cast<MetaEntry *>(sm + lay.off_meta);
  const uint32_t tmem_a = tmem;                                        // A slots: a_cols columns each
  const uint32_t tmem_d = tmem + lay.a_cols * static_cast<uint32_t>(na);  // D slots: NR columns each

  if (warp == 0) {
    // ================================================================ producer
    // The warp issues tiles in batches of nb, one tile per lane, so the
    // per-tile waits and copy issues run side by side; the q-record copies
    // of segments starting in a batch follow, in segment order, from lane 0.
    const int ns = lay.ns;
    // at most half the stages per batch, so the other half stays in flight
    // and no two tiles of a batch share a stage
    const int nb = min(8, ns / 2);
    const uint64_t pol_stream = ptx::policy_evict_first();   // keys are read once
    int issued = 0, last_seg0 = -1, last_seg1 = -1;   // latest record copied into each slot
    bool qrec_ready = false;
    for (int base = 0; base < n_tiles; base += nb) {
      const int i = base + lane;
      const bool act = lane < nb && i < n_tiles;
      const int s = i % ns, r = i & (kR - 1);
      bool ok = true;
      int seg = 0, tq = 0;
      if (act) {
        ok = ptx::mbar_wait(bar(B_EMPTY_RAW + s), (static_cast<uint32_t>(i / ns) & 1u) ^ 1u, abort_flag, kTimeoutNs);
        ok = ok && ptx::mbar_wait(bar(B_META_FULL + r), static_cast<uint32_t>(i / kR) & 1u, abort_flag, kTimeoutNs);
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      if (act) {
        const MetaEntry &m = sMeta[r];
        seg = m.seg;
        tq = m.t;
        const uint32_t mask = m.mask;
        const int s0 = m.s0, lb0 = m.lb0, nblk = m.nblk;
        // a block's copies: its keys within the tile (rows lo .. hi of the
        // tile's key range); a debug-bounds build checks them against the pool
        auto copy_ok = [&](int b) {
          const int blk0 = (lb0 + b) << lay.epb_shift;
          const int lo = max(s0, blk0), hi = min(s0 + kTileKeys, blk0 + p.epb);
          const long long row0 = (static_cast<long long>(m.phys[b]) << lay.epb_shift) + (lo - blk0);
          return IDX_IN_BOUNDS(row0 >= 0 && row0 + (hi - lo) <= static_cast<long long>(p.P) * p.epb &&
                                   hi - s0 <= kTileKeys,
                               p.dev_status);
        };
        uint32_t bytes = 0, copied = 0;   // copied: bit b, block b's copies are issued
        for (int b = 0; b < nblk; ++b) {
          if (!((mask >> b) & 1u) || !copy_ok(b)) continue;
          const int blk0 = (lb0 + b) << lay.epb_shift;
          bytes += static_cast<uint32_t>(min(s0 + kTileKeys, blk0 + p.epb) - max(s0, blk0)) * 72u;
          copied |= 1u << b;
        }
        const uint32_t full = bar(B_FULL_RAW + s);
        uint8_t *stage = sRaw + static_cast<size_t>(s) * kStageBytes;
        if (bytes == 0) {
          ptx::mbar_arrive(full);
        } else {
          ptx::mbar_arrive_expect_tx(full, bytes);
          for (int b = 0; b < nblk; ++b) {
            if (!((copied >> b) & 1u)) continue;
            const int blk0 = (lb0 + b) << lay.epb_shift;
            const int lo = max(s0, blk0), hi = min(s0 + kTileKeys, blk0 + p.epb);
            const long long row0 = (static_cast<long long>(m.phys[b]) << lay.epb_shift) + (lo - blk0);
            const int dst_row = lo - s0;
            for (int rr = 0; rr < hi - lo; rr += lay.box_rows) {
              const uint32_t dst = ptx::smem_addr(stage + (dst_row + rr) * 64);
              asm volatile(
                  "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                  " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
                  "l"(reinterpret_cast<uint64_t>(&tmap_nib)), "r"(0), "r"(static_cast<int>(row0 + rr)),
                  "r"(full), "l"(pol_stream)
                  : "memory");
            }
            ptx::bulk_g2s_hint(ptx::smem_addr(stage + kScaleOff + dst_row * 8), p.key_scale + row0 * 8,
                               static_cast<uint32_t>(hi - lo) * 8u, full, pol_stream);
          }
        }
      }
      issued = min(base + nb, n_tiles);
      // Segments starting in this batch: copy q[t]'s B-operand record into
      // slot (ordinal mod nseg) once that slot's previous segment is done
      // with it. The batch's tiles are already on their way, so the waits
      // cannot hold up the segment they wait for.
      uint32_t segs = __ballot_sync(0xFFFFFFFFu, act && seg != 0);
      bool seg_ok = true;
      while (segs) {
        const int L = __ffs(segs) - 1;
        segs &= segs - 1;
        const int ord = __shfl_sync(0xFFFFFFFFu, seg, L) - 1, t_seg = __shfl_sync(0xFFFFFFFFu, tq, L);
        if (lane == 0) {
          const int ss = ord % nseg;
          const uint32_t ph = static_cast<uint32_t>(ord / nseg) & 1u;
          seg_ok = ptx::mbar_wait(bar(B_SEG_BFREE + ss), ph ^ 1u, abort_flag, kTimeoutNs) &&
                   ptx::mbar_wait(bar(B_SEG_WFREE + ss), ph ^ 1u, abort_flag, kTimeoutNs);
          if (seg_ok) {
            if (!qrec_ready) {
              ptx::wait_prior_grid();  // the records are written by the kernel launched just before
              qrec_ready = true;
            }
            const uint32_t sfull = bar(B_SEG_FULL + ss);
            ptx::mbar_arrive_expect_tx(sfull, lay.rec_bytes);
            ptx::bulk_g2s(ptx::smem_addr(sB + ss * lay.rec_smem), qrec + static_cast<size_t>(t_seg) * lay.rec_bytes,
                          lay.rec_bytes, sfull);
            if (ss == 0) last_seg0 = ord; else last_seg1 = ord;
          }
        }
        if (!__all_sync(0xFFFFFFFFu, __shfl_sync(0xFFFFFFFFu, seg_ok, 0))) break;
      }
      if (!__shfl_sync(0xFFFFFFFFu, seg_ok, 0)) break;
    }
    // Never leave with copies in flight: the last ns tile stages (one per
    // lane) and the latest record of each slot (an earlier one was waited for
    // before its slot's reuse).
    volatile int no_abort = 0;
    if (lane < ns) {
      const int i = issued - ns + lane;
      if (i >= 0)
        ptx::mbar_wait(bar(B_FULL_RAW + i % ns), static_cast<uint32_t>(i / ns) & 1u, &no_abort, kDrainNs);
    }
    const int ls0 = __shfl_sync(0xFFFFFFFFu, last_seg0, 0), ls1 = __shfl_sync(0xFFFFFFFFu, last_seg1, 0);
    const int last_rec = (lane == 0) ? ls0 : ls1;
    if ((lane == 0 || lane == 1) && last_rec >= 0)
      ptx::mbar_wait(bar(B_SEG_FULL + last_rec % nseg), static_cast<uint32_t>(last_rec / nseg) & 1u, &no_abort,
                     kDrainNs);
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    // The whole warp walks the tiles in lockstep; one elected lane issues.
    // Descriptors are built once per segment so the issue loop is nothing
    // but tcgen05.mma instructions.
    Walker<kRows> w;
    w.init(p, lay, t0, j0);
    const uint32_t idesc = kFp4 ? ptx::idesc_mxf4nvf4(128, NR) : ptx::idesc_f16_f32(128, NR);
    bool need_lo = false;
    uint64_t bdh[8], bdl[8];
    Ring ra, rd, rs, rraw;
    rs.idx = -1;  // advanced at each segment start
    int ss = 0;
    bool any_mma = false;
#ifdef IDX_TEST_STALL
    // Failure-path test builds only: CTA 0 first waits for a barrier nothing
    // ever arrives on, so its wait gives up, raises the abort flag and the
    // whole CTA takes the abort-and-drain path.
    if (blockIdx.x == 0) ptx::mbar_wait(bar(B_NEVER), 0u, abort_flag, kTimeoutNs);
#endif
    for (int i = 0; i < n_tiles; ++i, w.next(p, lay), ra.next(na), rd.next(nd), rraw.next(lay.ns)) {
      const bool seg_start = (i == 0) || (w.j == 0);
      const bool seg_end = (i == n_tiles - 1) || (w.j == w.nt - 1);
      bool ok = true;
      if (seg_start) {
        if (i > 0) rs.next(nseg); else rs.idx = 0;
        ss = rs.idx;
        ok = ptx::mbar_wait(bar(B_SEG_FULL + ss), rs.phase, abort_flag, kTimeoutNs);
        const uint8_t *slot = sB + ss * lay.rec_smem;
        if constexpr (kFp4) {   // q codes: K steps of 64 elements = 32 bytes into each 64-byte row
          bdh[0] = ptx::sdesc_sw64(ptx::smem_addr(slot));
          bdh[1] = ptx::sdesc_sw64(ptx::smem_addr(slot) + 32);
        } else {
          const int *flags = reinterpret_cast<const int *>(slot + lay.rec_flags);
          int f = 0;
          for (int h = lane; h < NR; h += 32) f |= flags[h];
          need_lo = __any_sync(0xFFFFFFFFu, f != 0);
          const uint32_t bh = ptx::smem_addr(slot);
          const uint32_t bl = ptx::smem_addr(slot + b_bytes);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t boff = (k >> 2) * (NR * 128) + (k & 3) * 32;
            bdh[k] = ptx::sdesc_sw128(bh + boff);
            bdl[k] = ptx::sdesc_sw128(bl + boff);
          }
        }
      }
      const int a = ra.idx, d = rd.idx, s = rraw.idx;
      ok = ok && ptx::mbar_wait(bar(B_FULL_A + a), ra.phase, abort_flag, kTimeoutNs);
      ok = ok && ptx::mbar_wait(bar(B_EMPTY_D + d), rd.phase ^ 1u, abort_flag, kTimeoutNs);
      // NVFP4-q: the MMA reads the stage itself (the decoders waited for it too)
      if (kFp4) ok = ok && ptx::mbar_wait(bar(B_FULL_RAW + s), rraw.phase, abort_flag, kTimeoutNs);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t dt = tmem_d + d * NR, at = tmem_a + a * lay.a_cols;
      if (ptx::elect_one()) {
        if constexpr (kFp4) {
          // A: the stage's 128 key rows of 64 bytes; scale slot: key scales
          // (columns 0-7), q scales (8-15), four columns per K step
          const uint32_t sa = ptx::smem_addr(sRaw + static_cast<size_t>(s) * kStageBytes);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            ptx::mma_ss_nvf4(dt, ptx::sdesc_sw64(sa + 32 * c), bdh[c], idesc, at + 4 * c, at + 8 + 4 * c,
                             c > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) ptx::mma_ts_f16(dt, at + 8 * k, bdh[k], idesc, k > 0 ? 1u : 0u);
          if (need_lo) {
#pragma unroll
            for (int k = 0; k < 8; ++k) ptx::mma_ts_f16(dt, at + 8 * k, bdl[k], idesc, 1u);
          }
        }
        ptx::mma_commit(bar(B_EMPTY_A + a));
        ptx::mma_commit(bar(B_FULL_D + d));
        if (kFp4) ptx::mma_commit(bar(B_EMPTY_RAW + s));
        if (seg_end) ptx::mma_commit(bar(B_SEG_BFREE + ss));
      }
      __syncwarp();
      any_mma = true;
    }
    // Never leave with MMAs in flight (the epilogue waits for each of them,
    // but not after an abort): tensor memory is freed after this.
    if (any_mma) {
      volatile int no_abort = 0;
      if (ptx::elect_one()) ptx::mma_commit(bar(B_DRAIN));
      __syncwarp();
      ptx::mbar_wait(bar(B_DRAIN), 0u, &no_abort, kDrainNs);
    }
  } else if (warp < kEpiWarp0) {
    // ============================================================== decoders
    if constexpr (kFp4) {
      // NVFP4-q: nothing to decode. Each tile's key scales (from the stage) and
      // its segment's q scales (from the record) go into the tile's
      // tensor-memory scale slot: word j of K step c holds the four scales of
      // row lane + 32 j, columns 4c + j (keys) and 8 + 4c + j (q). Every warp
      // writes the same words into its own 32-lane quarter.
      const uint32_t lane_q = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      Walker<kRows> w;
      w.init(p, lay, t0, j0);
      Ring rraw, ra, rs;
      int ss = 0;
      for (int i = 0; i < n_tiles; ++i, w.next(p, lay), rraw.next(lay.ns), ra.next(na)) {
        const int s = rraw.idx, a = ra.idx;
        bool ok = true;
        if (i == 0 || w.j == 0) {
          if (i > 0) rs.next(nseg);
          ss = rs.idx;
          ok = ptx::mbar_wait(bar(B_SEG_FULL + ss), rs.phase, abort_flag, kTimeoutNs);
        }
        ok = ok && ptx::mbar_wait(bar(B_FULL_RAW + s), rraw.phase, abort_flag, kTimeoutNs);
        ok = ok && ptx::mbar_wait(bar(B_EMPTY_A + a), ra.phase ^ 1u, abort_flag, kTimeoutNs);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        ptx::tc_fence_after();
        const uint8_t *stage = sRaw + static_cast<size_t>(s) * kStageBytes;
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(sB + ss * lay.rec_smem + lay.sfb_off);
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint2 sc = *reinterpret_cast<const uint2 *>(stage + kScaleOff + (lane + 32 * j) * 8);
          v[j] = sc.x;       // K step 0: groups 0-3 of key row lane + 32 j
          v[4 + j] = sc.y;   // K step 1: groups 4-7
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) v[8 + k] = qs[k * 32 + lane];
        ptx::tmem_st16(tmem_a + a * lay.a_cols + lane_q, v);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(B_FULL_A + a));
      }
    } else {
      const int row = 32 * (warp & 3) + lane;    // the TMEM lane this thread writes
      const int rsw = (row >> 1) & 3;            // 64-byte swizzle of this row's chunks
      constexpr int kHalves = 8 / kDecWarps;     // 64-element halves of the row per warp
      const int half0 = (kDecWarps == 8) ? ((warp - 2) >> 2) : 0;
      Ring rraw, ra;
      for (int i = 0; i < n_tiles; ++i, rraw.next(lay.ns), ra.next(na)) {
        const int s = rraw.idx, a = ra.idx;
        bool ok = ptx::mbar_wait(bar(B_FULL_RAW + s), rraw.phase, abort_flag, kTimeoutNs);
        ok = ok && ptx::mbar_wait(bar(B_EMPTY_A + a), ra.phase ^ 1u, abort_flag, kTimeoutNs);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        ptx::tc_fence_after();
        const uint8_t *stage = sRaw + static_cast<size_t>(s) * kStageBytes;
        const uint2 scw = *reinterpret_cast<const uint2 *>(stage + kScaleOff + row * 8);
        const uint32_t taddr = tmem_a + a * 64 + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          const int half = half0 + hh;
          uint32_t v[32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = half * 2 + cc;  // 16-byte chunk: elements 32c .. 32c+31, groups 2c, 2c+1
            const uint4 raw = *reinterpret_cast<const uint4 *>(stage + row * 64 + ((c ^ rsw) * 16));
            const uint32_t sc2 = ptx::e4m3x2_to_f16x2(((c < 2 ? scw.x : scw.y) >> (16 * (c & 1))) & 0xFFFFu);
            const uint32_t s_lo = __byte_perm(sc2, 0, 0x1010), s_hi = __byte_perm(sc2, 0, 0x3232);
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t e[4];
              ptx::e2m1x8_to_f16x2x4(wv[q4], e);
#pragma unroll
              for (int bb = 0; bb < 4; ++bb) v[cc * 16 + q4 * 4 + bb] = ptx::hmul2(e[bb], q4 < 2 ? s_lo : s_hi);
            }
          }
          ptx::tmem_st32(taddr + half * 32, v);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(bar(B_FULL_A + a));
          ptx::mbar_arrive(bar(B_EMPTY_RAW + s));
        }
      }
    }
  } else if (warp == kResolverWarp) {
    // ============================================================== resolver
    // Resolves block-table entries and global scales for batches of 32 blocks
    // at once (one per lane), so the two dependent global loads per block
    // overlap across the batch instead of serialising the TMA producer.
    const int bpt = lay.bpt;                 // blocks per full tile (epb a power of two)
    const int tpb = 32 / bpt;                // tiles per batch
    const int d = lane / bpt, b = lane % bpt;
    Walker<kRows> w;
    w.init(p, lay, t0, j0);
    int seg_base = 0;  // segments started before this batch
    for (int base = 0; base < n_tiles; base += tpb) {
      const int i = base + d;
      const bool tile_ok = i < n_tiles;
      Walker<kRows> wl = w;
      for (int x = 0; x < d && tile_ok; ++x) wl.next(p, lay);
      int L = 0, s0 = 0, lb0 = 0, nblk = 0, phys = -1, l0 = 0, l1 = 0;
      float g = 0.0f;
      bool blk_ok = false, pv = false;
      if (tile_ok) {
        l0 = row_len(p, wl.t * kRows);
        l1 = (kRows > 1 && wl.t * kRows + 1 < p.T) ? row_len(p, wl.t * kRows + 1) : 0;
        L = max(l0, l1);
        s0 = wl.j * kTileKeys;
        const int s_end = min(s0 + kTileKeys, L);
        lb0 = s0 >> lay.epb_shift;
        nblk = ((s_end - 1) >> lay.epb_shift) - lb0 + 1;
        blk_ok = b < nblk;
        if (blk_ok) {
          phys = p.block_table[static_cast<long long>(wl.t) * p.bt_stride + lb0 + b];
          pv = phys >= 0 && phys < p.P;
          if (pv) g = p.key_gscale[phys];
        }
      }
      if (blk_ok && !pv && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_BAD_BLOCK);
      const uint32_t valid_bits = __ballot_sync(0xFFFFFFFFu, pv);
      const bool starts = tile_ok && b == 0 && (i == 0 || wl.j == 0);
      const uint32_t start_bits = __ballot_sync(0xFFFFFFFFu, starts);
      const int ord = seg_base + __popc(start_bits & lanemask_lt());
      seg_base += __popc(start_bits);
      const int r = i & (kR - 1);   // kR is a power of two
      bool ok = true;
      if (tile_ok && b == 0)
        ok = ptx::mbar_wait(bar(B_META_EMPTY + r), (static_cast<uint32_t>(i / kR) & 1u) ^ 1u, abort_flag,
                            kTimeoutNs);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      MetaEntry &m = sMeta[r];
      if (blk_ok) {
        m.phys[b] = phys;
        m.g[b] = g;
      }
      if (tile_ok && b == 0) {
        m.mask = (valid_bits >> (d * bpt)) & ((bpt == 32) ? 0xFFFFFFFFu : ((1u << bpt) - 1u));
        m.lb0 = lb0;
        m.s0 = s0;
        m.nblk = nblk;
        m.t = wl.t;
        m.seg = starts ? ord + 1 : 0;
        m.len[0] = l0;
        m.len[1] = l1;
      }
      __syncwarp();
      if (tile_ok && b == 0) ptx::mbar_arrive(bar(B_META_FULL + r));
      for (int x = 0; x < tpb; ++x) w.next(p, lay);
    }
  } else {
    // ============================================================== epilogue
    // lay.ne (at most kEpiGroups, at most one per D slot) groups of four
    // warps take tiles in turn (one group's tile takes longer than the MMA of
    // one tile); the warps of any other group only keep count. Every warp still walks every
    // tile: it waits for each segment's q record and signals when it is done
    // with each segment's w', so a slot is reused only after every group is
    // done with it.
    const int row = 32 * (warp & 3) + lane;    // the TMEM lane (key row) this thread reads
    const int grp = (warp - kEpiWarp0) >> 2;
    Walker<kRows> w;
    w.init(p, lay, t0, j0);
    int ss = 0;
    Ring rd, rm, rs, rg;   // rg.idx: the group whose tile this is
    for (int i = 0; i < n_tiles; ++i, w.next(p, lay), rd.next(nd), rm.next(kR), rg.next(lay.ne)) {
      const bool seg_start = (i == 0) || (w.j == 0);
      const bool seg_end = (i == n_tiles - 1) || (w.j == w.nt - 1);
      bool ok = true;
      if (seg_start) {
        if (i > 0) rs.next(nseg);
        ss = rs.idx;
        ok = ptx::mbar_wait(bar(B_SEG_FULL + ss), rs.phase, abort_flag, kTimeoutNs);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
      }
      if (rg.idx != grp) {       // another group's tile
        if (seg_end) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(B_SEG_WFREE + ss));
        }
        continue;
      }
      const int d = rd.idx, r = rm.idx;
      ok = ok && ptx::mbar_wait(bar(B_FULL_D + d), rd.phase, abort_flag, kTimeoutNs);
      ok = ok && ptx::mbar_wait(bar(B_META_FULL + r), rm.phase, abort_flag, kTimeoutNs);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;  // warp-uniform exit before the .aligned TMEM loads
      ptx::tc_fence_after();
      const int s_key = w.j * kTileKeys + row;
      const int b = (s_key >> lay.epb_shift) - sMeta[r].lb0;
      const bool blk_ok = b < kMaxBlocksPerTile && ((sMeta[r].mask >> b) & 1u);
      const float g = (b < kMaxBlocksPerTile) ? sMeta[r].g[b] : 0.0f;
      const int len0 = sMeta[r].len[0], len1 = sMeta[r].len[1];
      const float *wq = reinterpret_cast<const float *>(sB + ss * lay.rec_smem + lay.rec_w);  // w'_n
      const uint32_t taddr = tmem_d + d * NR + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {    // rows of the group: head rows rr Npad .. rr Npad + Npad - 1
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // eight independent chains
        for (int c0 = rr * Npad; c0 < (rr + 1) * Npad; c0 += 32) {   // Npad is a multiple of 32
          uint32_t v[32];
          __syncwarp();  // the per-row sign branch below must not leave the warp split at these loads
          ptx::tmem_ld32(taddr + c0, v);
          ptx::tmem_wait_ld();
          if (c0 + 32 >= NR) {   // every accumulator column is in registers: hand back the slots
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(bar(B_EMPTY_D + d));
              ptx::mbar_arrive(bar(B_META_EMPTY + r));
            }
          }
          const float4 *w4 = reinterpret_cast<const float4 *>(wq + c0);
          if (g >= 0.0f) {          // relu(g a) = g max(a, 0)
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 ww = w4[e >> 2];
              float *ac = acc + ((e >> 2) & 1) * 4;
              ac[0] = fmaf(ww.x, fmaxf(__uint_as_float(v[e + 0]), 0.0f), ac[0]);
              ac[1] = fmaf(ww.y, fmaxf(__uint_as_float(v[e + 1]), 0.0f), ac[1]);
              ac[2] = fmaf(ww.z, fmaxf(__uint_as_float(v[e + 2]), 0.0f), ac[2]);
              ac[3] = fmaf(ww.w, fmaxf(__uint_as_float(v[e + 3]), 0.0f), ac[3]);
            }
          } else {                  // relu(g a) = g min(a, 0)
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 ww = w4[e >> 2];
              float *ac = acc + ((e >> 2) & 1) * 4;
              ac[0] = fmaf(ww.x, fminf(__uint_as_float(v[e + 0]), 0.0f), ac[0]);
              ac[1] = fmaf(ww.y, fminf(__uint_as_float(v[e + 1]), 0.0f), ac[1]);
              ac[2] = fmaf(ww.z, fminf(__uint_as_float(v[e + 2]), 0.0f), ac[2]);
              ac[3] = fmaf(ww.w, fminf(__uint_as_float(v[e + 3]), 0.0f), ac[3]);
            }
          }
        }
        const float sum = ((acc[0] + acc[4]) + (acc[1] + acc[5])) + ((acc[2] + acc[6]) + (acc[3] + acc[7]));
        const int t = w.t * kRows + rr;
        if (s_key < (rr == 0 ? len0 : len1) && IDX_IN_BOUNDS(t < p.T && s_key < ld, p.dev_status)) {
          // (an absent row or a bad length has length 0)
          const float sc = __fadd_rn(g * sum, 0.0f);
          scores[static_cast<long long>(t) * ld + s_key] = blk_ok ? sc : -INFINITY;
          // the selection's first digit: top 12 bits of the order-preserving key
          if (blk_ok && sc != -INFINITY)   // exactly the keys the selection will see
            atomicAdd(hist + static_cast<size_t>(t) * kScoreBins + (float_order(sc) >> 20), 1u);
        }
      }
      if (seg_end) {             // this warp is done with the segment's w'
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(B_SEG_WFREE + ss));
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && misc[M_ABORT] && p.dev_status) atomicOr(p.dev_status, IDX_STATUS_TIMEOUT);
}

// ------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

bool make_layout(const ScoreParams &p, TcLayout *out) {
  TcLayout l{};
  l.Npad = round_up(p.H, 32);
  if (l.Npad > 256) return false;
  l.fp4 = (p.q_format == IDX_Q_NVFP4) ? 1 : 0;
  if (l.fp4) {
    // head rows in multiples of 64 (MMA N of 64 or 128); the q scale slot
    // covers 128 head rows
    l.Npad = round_up(p.H, 64);
    if (l.Npad > 128) return false;
  }
  // Row pairs share one decoded key tile (one MMA of N = 2 Npad) when every
  // row reads the same block table.
  l.R = (p.bt_stride == 0 && p.T >= 2 && l.Npad <= 64) ? 2 : 1;
  l.NR = l.R * l.Npad;
  l.nq = (p.T + l.R - 1) / l.R;
  l.nseg = (l.NR <= 128) ? 2 : 1;
  // Tensor memory (512 columns): na A slots of 64 columns (128 keys x 128 f16)
  // and nd D slots of Npad columns (128 keys x Npad f32 accumulators); more
  // slots let the decoders, the MMA and the epilogue run further apart.
  // NVFP4-q: an A slot holds only the tile's scale factors (16 columns).
  l.a_cols = l.fp4 ? 16u : 64u;
  l.na = (l.fp4 || l.NR <= 64) ? 4 : 2;
  l.nd = (512 - static_cast<int>(l.a_cols) * l.na) / l.NR;
  if (l.nd > kMaxSlots) l.nd = kMaxSlots;
  if (l.nd < 1) return false;
  // Epilogue groups in use: at most one per D slot. A group waits for the D
  // slot of its tile i with the slot's phase parity; the tile nd before it
  // must already be complete for that parity to be unambiguous, which the
  // group's own previous tile (i - ne) guarantees when ne <= nd.
  l.ne = (l.nd < kEpiGroups) ? l.nd : kEpiGroups;
  if (p.epb < 16 || (p.epb & (p.epb - 1)) != 0) return false;  // power-of-two blocks of >= 16 keys
  l.box_rows = p.epb < 128 ? p.epb : 128;
  l.bpt = p.epb < 128 ? 128 / p.epb : 1;
  l.epb_shift = 0;
  while ((1 << l.epb_shift) < p.epb) ++l.epb_shift;
  // B-operand records first (1 KB-aligned slots), then the raw stages (1 KB
  // multiples, as many as fit), then the small tables.
  if (l.fp4) {
    l.b_bytes = static_cast<uint32_t>(l.NR) * 64u;   // E2M1 codes
    l.sfb_off = l.b_bytes;                         // then 1 KB of scale words
    l.rec_w = l.sfb_off + 1024u;
  } else {
    l.b_bytes = static_cast<uint32_t>(l.NR) * 256u;
    l.sfb_off = 0;
    l.rec_w = 2u * l.b_bytes;
  }
  l.rec_flags = l.rec_w + static_cast<uint32_t>(l.NR) * 4u;
  l.rec_bytes = (l.rec_flags + static_cast<uint32_t>(l.NR) * 4u + 127u) & ~127u;
  l.rec_smem = (l.rec_bytes + 1023u) & ~1023u;
  l.off_b = 0;
  const uint32_t b_total = static_cast<uint32_t>(l.nseg) * l.rec_smem;
  const uint32_t tail = kR * sizeof(MetaEntry) + ((B_COUNT * 8 + 15) & ~15u) + ((kMiscBytes + 15) & ~15u);
  const long long room = static_cast<long long>(kSmemLimit) - 1024 - b_total - tail;
  long long ns = room / kStageBytes;
  if (ns > kMaxNS) ns = kMaxNS;
  if (ns < 3) return false;
  l.ns = static_cast<int>(ns);
  uint32_t off = b_total;
  l.off_raw = off;
  off += static_cast<uint32_t>(l.ns) * kStageBytes;
  l.off_meta = off;
  off += kR * sizeof(MetaEntry);
  l.off_bar = off;
  off += B_COUNT * 8;
  off = (off + 15) & ~15u;
  l.off_misc = off;
  off += kMiscBytes;
  off = (off + 15) & ~15u;
  l.smem_bytes = off + 1024;
  *out = l;
  return true;
}

}  // namespace

bool score_tc_supported(const ScoreParams &p) {
  TcLayout l;
  if (static_cast<long long>(p.P) * p.epb >= (1LL << 31)) return false;  // TMA row coordinate is int32
  return p.D == 128 && p.keys_fp4 != nullptr && make_layout(p, &l) && get_encode() != nullptr;
}

size_t score_tc_workspace(const ScoreParams &p) {
  TcLayout lay;
  if (!make_layout(p, &lay)) return 0;
  return static_cast<size_t>(lay.nq) * lay.rec_bytes;
}

cudaError_t launch_score_tc(const ScoreParams &p, int num_ctas, void *qrec, uint32_t *hist, uint32_t *cand_cnt,
                            float *scores, long long ld, cudaStream_t stream) {
  TcLayout lay;
  if (!make_layout(p, &lay)) return cudaErrorNotSupported;
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(p.P) * static_cast<cuuint64_t>(p.epb)};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(lay.box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.keys_fp4), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  void (*kern)(const CUtensorMap, ScoreParams, TcLayout, const uint8_t *, uint32_t *, float *, long long) =
      lay.fp4 ? ((lay.R == 2) ? score_tc_kernel<2, true> : score_tc_kernel<1, true>)
              : ((lay.R == 2) ? score_tc_kernel<2, false> : score_tc_kernel<1, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(lay.smem_bytes));
  if (e != cudaSuccess) return e;
  uint8_t *rec = static_cast<uint8_t *>(qrec);
  if (lay.nq >= 2 * num_ctas)   // enough records to fill the GPU block by block
    qprep_kernel<<<static_cast<unsigned>(lay.nq), 256, 0, stream>>>(p, lay, rec, hist, cand_cnt);
  else
    qprep_rows_kernel<<<dim3(static_cast<unsigned>(lay.nq), static_cast<unsigned>(lay.NR / 8)), 256, 0, stream>>>(
        p, lay, rec, hist, cand_cnt);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // The scorer may launch while qprep_kernel runs: its producer waits for the
  // records (griddepcontrol.wait) only before the first record copy.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(num_ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = lay.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmap, p, lay, static_cast<const uint8_t *>(rec), hist, scores, ld);
}

namespace {

// The NVFP4-q mode's quantisation on its own, one warp per head row of 128:
// codes [rows, 64] bytes (low nibble = even element), scales [rows, 8] E4M3,
// gscale [rows] float32.
__global__ void __launch_bounds__(256) quantize_q_kernel(const float *__restrict__ q, long long rows,
                                                         uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                                                         float *__restrict__ gscale) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;   // whole warps
  const float4 x = reinterpret_cast<const float4 *>(q + row * 128)[lane];
  uint32_t c16, sc;
  float gq;
  nvfp4_quantize_lane(x, c16, sc, gq);
  reinterpret_cast<uint16_t *>(codes + row * 64)[lane] = static_cast<uint16_t>(c16);
  if ((lane & 3) == 0) scales[row * 8 + (lane >> 2)] = static_cast<uint8_t>(sc);
  if (lane == 0) gscale[row] = gq;
}

}  // namespace

cudaError_t launch_quantize_q_nvfp4(const float *q, long long rows, uint8_t *codes, uint8_t *scales, float *gscale,
                                    cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  quantize_q_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(q, rows, codes, scales, gscale);
  return cudaGetLastError();
}

}  // namespace idx
