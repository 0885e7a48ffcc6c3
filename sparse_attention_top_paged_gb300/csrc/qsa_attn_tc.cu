// qsa_attn_tc.cu — QSA prefill attention on the tcgen05 tensor cores, for G = 1,
// 2, 4 or 8 query heads per kv head and hd = 128 ("metrale_model_layers/layers/ops/qsa.rs",
// qsa_prefill_attn: per (row, query head) one softmax over every token of the
// row's selected complete blocks and over the incomplete tail, with K and V of
// the head's kv head read through the page table).
//
// Work item = (row, kv head); its tokens are numbered list-major (token t of
// selected block i is i * ratio + t; blocks that are not complete are
// skipped), then the tail, and cut into steps of 128 tokens. The kernel is
// persistent, one CTA per SM taking items blockIdx.x, blockIdx.x + gridDim.x,
// ... Its steps, laid end to end, flow through a ring of kStages shared-memory
// stages:
//   warps 10-21 three producer groups of four warps taking the steps in turn.
//               For each step a group looks up its 128 tokens (list entry,
//               then page), copies their K and V rows (256 bytes each) into
//               the stage with 16-byte asynchronous copies in the 128-byte
//               swizzled layout the MMAs read (two 16 KB halves of 64
//               dimensions, token t's half-row at t * 128 bytes; zero rows for
//               tokens that are missing), writes the step's Qs operand (q *
//               inv_sqrt_d of the G heads split into bf16 high parts, rows 0-7,
//               and low parts, rows 8-15, once per item: q keeps about 17
//               significant bits; rows of unused head slots are zero) and the
//               token mask. The copies arrive on the stage's barrier when they
//               land, so a group never waits on its own copies.
//   warp 8      score MMAs (tcgen05, kind::f16, bf16 operands, f32 in tensor
//               memory): S^T[128 tokens x 16] = K . Qs^T of step j into S slot
//               j % 2 (S = column h + column 8 + h), as soon as the stage is
//               full and the softmax of step j - 2 has left the slot.
//   warp 9      value MMAs: O^T[128 dims x 16] += V^T . P^T of step j once its
//               weights are written, V read in place as an MN-major operand
//               (the step's token rows are its K rows), into the item's O slot
//               (two, by item parity). Its commit frees the stage. With two
//               issuing warps a step's value MMAs never wait behind the issue
//               of the next step's scores.
//   warps 0-7   softmax: warp w owns tensor-memory lanes 32 (w % 4) .. + 31
//               (tokens of S, dimensions of O) for (G + 1) / 2 head slots. Each
//               head keeps a lazy reference maximum that moves only when a
//               score exceeds it by more than kLazy. Per step the warps write
//               the weights p = exp(S - ref), split into bf16 high and low
//               parts, as the value MMA's B operand (two P slots, a slot
//               reused once the value MMA two steps back is done) and take one
//               vote; only when some score broke its reference (an item's
//               first step, or a jump) do they exchange the heads' maxima over
//               the step, move the references, rescale the running sums and
//               the head's two output columns, and write the weights again. An
//               item's output, dimension d of head h = (column h + column 8 +
//               h) / sum, is written after the next item's first step, once
//               its last value MMA is done, so the tensor pipe does not drain
//               at each item's end.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace idx {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kMmaWarp = kComputeWarps;   // issues the score MMAs; the next warp the value MMAs
constexpr int kProdWarp0 = kMmaWarp + 2;
constexpr int kProdGroups = 3;
constexpr int kThreads = 32 * (kProdWarp0 + 4 * kProdGroups);
constexpr int kStages = 3;
constexpr int kTok = 128, kHd = 128;
constexpr int kGroup = 8;   // head slots of the MMAs (N = 16: high and low parts); G <= 8 of them are used
constexpr float kLazy = 8.0f;
// a stage: K rows, V rows (32 KB each), the Qs operand (16 rows x 128 dims), the token mask
constexpr uint32_t kOffK = 0, kOffV = 32768, kOffQ = 65536, kOffMask = 69632;
constexpr uint32_t kStageBytes = 70656;                  // 1 KB aligned
constexpr uint32_t kOffP = kStages * kStageBytes;        // two P slots: 16 rows x 128 tokens each
constexpr uint32_t kOffRed = kOffP + 2 * 4096;           // [4 lane quarters][8 heads] maxima, then 2 x sums
constexpr uint32_t kOffBar = kOffRed + 3 * 4 * kGroup * 4;
// per stage: full, empty; per slot (step parity): S^T written, weights written
constexpr int B_FULL = 0, B_EMPTY = kStages, B_S = 2 * kStages, B_P = 2 * kStages + 2, B_NEVER = 2 * kStages + 4,
              B_DRAIN = 2 * kStages + 5, B_COUNT = 2 * kStages + 7;   // B_DRAIN: one per MMA-issuing warp
constexpr uint32_t kOffMisc = kOffBar + 8 * B_COUNT;     // tensor-memory address, abort flag, bad-block flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;    // + slack to align the base to 1 KB
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
constexpr uint32_t kTmemCols = 64;   // S slots: columns 0-15, 16-31; O slots (item parity): 32-47, 48-63
// Every wait gives up after kWaitNs (2 s; failure-path test builds shorten it
// with IDX_WAIT_LIMIT_NS), raising the CTA's abort flag: the CTA then leaves
// with no copy or MMA in flight and the call reports IDX_STATUS_TIMEOUT.
#ifdef IDX_WAIT_LIMIT_NS
constexpr uint64_t kWaitNs = IDX_WAIT_LIMIT_NS;
#else
constexpr uint64_t kWaitNs = 2000000000ull;
#endif

// Shared-memory descriptor, 128-byte swizzle: K-major (lbo unused: 16) or
// MN-major (lbo = the stride between 64-element atoms along M or N); sbo =
// the stride between groups of 8 rows.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// kind::f16 instruction descriptor: f32 accumulator, bf16 A and B, M = 128,
// N = 16; A MN-major (transposed) when mn_a.
__host__ __device__ constexpr uint32_t idesc_bf16(bool mn_a) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (mn_a ? (1u << 15) : 0u) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t (&v)[1]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v[0]) : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, const uint32_t (&v)[1]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v[0]) : "memory");
}

__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t (&v)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_st2(uint32_t taddr, const uint32_t (&v)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(v[0]), "r"(v[1]) : "memory");
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}

// n consecutive columns of this warp's lanes (n = 1, 2 or 4)
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&v)[N]) {
  if constexpr (N == 1) tmem_ld1(taddr, v);
  else if constexpr (N == 2) tmem_ld2(taddr, v);
  else tmem_ld4(taddr, v);
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 1) tmem_st1(taddr, v);
  else if constexpr (N == 2) tmem_st2(taddr, v);
  else tmem_st4(taddr, v);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The barrier receives one arrival once every earlier asynchronous copy of
// this thread has landed (its initial count includes these arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Barrier 1 over the softmax warps; returns whether `ok` holds in every one of
// their threads.
__device__ __forceinline__ bool compute_sync_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n"
      " barrier.cta.red.and.pred b, 1, %2, a;\n selp.u32 %0, 1, 0, b;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok)), "n"(32 * kComputeWarps)
      : "memory");
  return r != 0;
}

// Barrier 1 over the softmax warps; returns how many of their threads have
// `pred` set.
__device__ __forceinline__ uint32_t compute_sync_count(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a;\n setp.ne.u32 a, %1, 0;\n barrier.cta.red.popc.u32 %0, 1, %2, a;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(32 * kComputeWarps)
      : "memory");
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// The byte offset of element (row, col) of a 128-byte-swizzled operand whose
// rows hold 64 bf16 elements and whose second 64 columns sit `half` bytes on.
__device__ __forceinline__ uint32_t sw128(int row, int col, uint32_t half) {
  return (col >> 6) * half + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2;
}

// floor(n / d) for n < 2^31 as (n m) >> s, with s = 31 + ceil(log2 d) and m =
// ceil(2^s / d) < 2^32: division by an invariant integer through multiplication
// (Granlund and Montgomery); m d - 2^s < d keeps the error below one for such n.
struct DivU {
  uint32_t m, s;
};
inline DivU div_magic(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  return DivU{static_cast<uint32_t>(((1ull << (31 + l)) + d - 1) / d), 31 + l};
}
__device__ __forceinline__ uint32_t divu(uint32_t n, DivU d) {
  return static_cast<uint32_t>((static_cast<unsigned long long>(n) * d.m) >> d.s);
}

struct Problem {
  const float *q;
  const uint16_t *kc, *vc;
  const int32_t *table, *lists;
  float *out;
  int n_pages, P;
  uint32_t first_pos, topk, ratio, block_size, nq, nkv;
  float inv_sqrt_d;
  DivU by_ratio, by_block;   // the token lookups' divisions (operands below 2^31)
};

// One item's token numbering: list tokens [0, n_list), then the tail. Items,
// positions and token numbers are 32-bit (the launch checks that they fit).
struct Item {
  uint32_t r, kvh, ncomp, n_list, tail0, n_virt;
  __device__ void set(const Problem &pr, uint32_t w) {
    r = w / pr.nkv;
    kvh = w - r * pr.nkv;
    const uint32_t p = pr.first_pos + r;
    ncomp = (p + 1) / pr.ratio;
    n_list = pr.topk * pr.ratio;
    tail0 = ncomp * pr.ratio;
    n_virt = n_list + (p + 1 - tail0);
  }
};

// The steps of a CTA in order: items blockIdx.x + i * gridDim.x with at least
// one token, 128 tokens at a time.
struct StepWalk {
  uint32_t w, items, base;
  Item it;
  bool valid;
  uint32_t par = 0;   // parity of the item's ordinal in the CTA's walk
  __device__ void seek(const Problem &pr) {   // from item w: the first one with tokens
    for (; w < items; w += gridDim.x, par ^= 1u) {
      it.set(pr, w);
      if (it.n_virt > 0) {
        base = 0;
        valid = true;
        return;
      }
    }
    valid = false;
  }
  __device__ void next(const Problem &pr) {
    base += kTok;
    if (base >= it.n_virt) {
      w += gridDim.x;
      par ^= 1u;
      seek(pr);
    }
  }
};

// A producer group (four warps, a token a thread): steps g, g + kProdGroups,
// ... of the CTA's walk; the groups' copies of consecutive steps overlap.
template <int G>
__device__ void producer(const Problem &pr, uint32_t items, unsigned char *sm, uint32_t s_base, int g, int pw,
                         int lane, volatile int *abort, int *bad_flag) {
  const int ptid = 32 * pw + lane;
  const uint32_t bar0 = s_base + kOffBar;
  StepWalk sw;
  sw.w = blockIdx.x;
  sw.items = items;
  sw.seek(pr);
  for (int i = 0; i < g && sw.valid; ++i) sw.next(pr);
  bool bad = false;
  uint32_t q_item = 0xFFFFFFFFu;   // the item whose Qs share this thread holds
  // this thread's share of the item's Qs operand: dimension pairs x = ptid + 128 i
  // (head x / 64, dimensions 2 (x % 64) and + 1), bf16 high and low parts
  uint32_t qhi[4] = {0u, 0u, 0u, 0u}, qlo[4] = {0u, 0u, 0u, 0u};
  for (uint32_t j = g; sw.valid; j += kProdGroups) {
    const int s = static_cast<int>(j % kStages);
    const uint32_t par = static_cast<uint32_t>((j / kStages) & 1);
    const bool q_new = sw.w != q_item;
    if (q_new) {   // the group's first step of an item: its q rows, scaled and split once
      q_item = sw.w;
      float2 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int x = ptid + 128 * i, h = x >> 6, d = 2 * (x & 63);
        v[i] = h < G ? *reinterpret_cast<const float2 *>(pr.q + (static_cast<long long>(sw.it.r) * pr.nq + sw.it.kvh * G + h) * kHd + d)
                     : make_float2(0.0f, 0.0f);   // unused head slots: zero rows
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a0 = v[i].x * pr.inv_sqrt_d, a1 = v[i].y * pr.inv_sqrt_d;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a0, a1);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a0 - __low2float(hi), a1 - __high2float(hi));   // exact differences
        qhi[i] = *reinterpret_cast<const uint32_t *>(&hi);
        qlo[i] = *reinterpret_cast<const uint32_t *>(&lo);
      }
    }
    // this thread's token (list entry, then page), before the stage is free: its cache
    // row (page, slot, kv head), 128 elements each, or -1
    int crow = -1;
    {
      const uint32_t v = sw.base + ptid;
      uint32_t pos = 0;
      bool has = false;
      if (v < sw.it.n_list) {
        const uint32_t bi = divu(v, pr.by_ratio);
        const int b = pr.lists[static_cast<long long>(sw.it.r) * pr.topk + bi];
        has = b >= 0 && static_cast<uint32_t>(b) < sw.it.ncomp;
        pos = static_cast<uint32_t>(b) * pr.ratio + (v - bi * pr.ratio);
      } else if (v < sw.it.n_virt) {
        has = true;
        pos = sw.it.tail0 + (v - sw.it.n_list);
      }
      if (has) {
        const uint32_t pg = divu(pos, pr.by_block);
        const int page = pg < static_cast<uint32_t>(pr.n_pages) ? pr.table[pg] : -1;
        if (page < 0 || page >= pr.P)
          bad = true;
        else
          crow = static_cast<int>((static_cast<uint32_t>(page) * pr.block_size + (pos - pg * pr.block_size)) * pr.nkv +
                                  sw.it.kvh);
      }
    }
    const uint32_t live = __ballot_sync(0xFFFFFFFFu, crow >= 0);
    if (!ptx::mbar_wait(bar0 + 8 * (B_EMPTY + s), par ^ 1u, abort, kWaitNs)) break;
    unsigned char *st = sm + s * kStageBytes;
    const uint32_t st_a = s_base + s * kStageBytes;
    if (lane == 0) reinterpret_cast<uint32_t *>(st + kOffMask)[pw] = live;
    // a half-warp copies one token's 256-byte K row and V row (16 lanes x 16 bytes)
    const uint16_t *kc_l = pr.kc + 8 * (lane & 15), *vc_l = pr.vc + 8 * (lane & 15);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = 2 * i + (lane >> 4), c = lane & 15;
      const int src = __shfl_sync(0xFFFFFFFFu, crow, t);
      const uint32_t o = sw128(32 * pw + t, 8 * c, 16384);
      if (src >= 0) {
        cp_async16(st_a + kOffK + o, kc_l + static_cast<long long>(src) * kHd);
        cp_async16(st_a + kOffV + o, vc_l + static_cast<long long>(src) * kHd);
      } else {   // no token: zero rows, so the value sum sees finite values
        *reinterpret_cast<uint4 *>(st + kOffK + o) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(st + kOffV + o) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // (group g fills stage g only: the stage still holds this item's Qs from the
    // group's previous step unless the item changed)
    static_assert(kProdGroups == kStages, "a group owns its stage");
    if (q_new) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int x = ptid + 128 * i, h = x >> 6, d = 2 * (x & 63);
        *reinterpret_cast<uint32_t *>(st + kOffQ + sw128(h, d, 2048)) = qhi[i];
        *reinterpret_cast<uint32_t *>(st + kOffQ + sw128(8 + h, d, 2048)) = qlo[i];
      }
    }
    cp_async_arrive(bar0 + 8 * (B_FULL + s));   // when this thread's copies have landed
    ptx::mbar_arrive(bar0 + 8 * (B_FULL + s));  // its plain stores (release)
    for (int i = 0; i < kProdGroups && sw.valid; ++i) sw.next(pr);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (bad) *bad_flag = 1;
}

// The MMA warp's S^T for step j (its stage is full): stage j % kStages, S slot
// j & 1. The whole warp calls it (operands stay warp-uniform); one lane issues.
__device__ __forceinline__ void issue_scores(uint32_t s_base, uint32_t tmem, uint32_t j) {
  const uint32_t st_a = s_base + static_cast<uint32_t>(j % kStages) * kStageBytes;
  const uint32_t d = tmem + 16 * static_cast<uint32_t>(j & 1);
  if (ptx::elect_one()) {
    ptx::fence_proxy_async_smem();   // the producers' plain and copied stores, to the tensor cores
    ptx::tc_fence_after();
#pragma unroll
    for (int k = 0; k < 8; ++k)
      mma_ss(d, sdesc(st_a + kOffK + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
             sdesc(st_a + kOffQ + (k >> 2) * 2048 + (k & 3) * 32, 16, 1024), idesc_bf16(false), k > 0 ? 1u : 0u);
    ptx::mma_commit(s_base + kOffBar + 8 * (B_S + static_cast<int>(j & 1)));
  }
  __syncwarp();
}

// The MMA warp's O^T += V^T . P^T for step j (its weights are written) into the
// item's O slot; its commit frees the stage.
__device__ __forceinline__ void issue_values(uint32_t s_base, uint32_t tmem, uint32_t j, bool first, uint32_t oslot) {
  const uint32_t st_a = s_base + static_cast<uint32_t>(j % kStages) * kStageBytes;
  const uint32_t p_a = s_base + kOffP + 4096u * static_cast<uint32_t>(j & 1);
  if (ptx::elect_one()) {
    ptx::fence_proxy_async_smem();   // the V rows (their landing was seen by the softmax warps)
    ptx::tc_fence_after();
#pragma unroll
    for (int k = 0; k < 8; ++k)
      mma_ss(tmem + 32 + oslot, sdesc(st_a + kOffV + k * 2048, 16384, 1024),
             sdesc(p_a + (k >> 2) * 2048 + (k & 3) * 32, 16, 1024), idesc_bf16(true), (!first || k > 0) ? 1u : 0u);
    ptx::mma_commit(s_base + kOffBar + 8 * (B_EMPTY + static_cast<int>(j % kStages)));
  }
  __syncwarp();
}

// After a wait gave up: the MMA warp's own MMAs retire before the CTA frees
// tensor memory (a commit tracks every earlier MMA of the issuing thread; the
// wait on it is bounded too).
__device__ __forceinline__ void drain_mmas(uint32_t bar) {
  if (ptx::elect_one()) ptx::mma_commit(bar);
  __syncwarp();
  volatile int no_abort = 0;
  ptx::mbar_wait(bar, 0u, &no_abort, kWaitNs);
}

__device__ __forceinline__ uint32_t full_bar(uint32_t bar0, uint32_t j) {
  return bar0 + 8 * (B_FULL + static_cast<int>(j % kStages));
}

// 22 warps (24 for register allocation, in groups of 4): at most 80 registers a thread
template <int G>
__global__ void __maxnreg__(80) qsa_prefill_attn_tc_kernel(Problem pr, uint32_t items,
                                                                          int32_t *dev_status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // aligned by pointer arithmetic on the shared array, so accesses through sm stay shared-space ones
  unsigned char *sm = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  float *red = reinterpret_cast<float *>(sm + kOffRed);   // maxima [4][8], sums [2][4][8]
  uint32_t *tmem_p = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  int *bad_flag = reinterpret_cast<int *>(sm + kOffMisc + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t s_base = ptx::smem_addr(sm), bar0 = s_base + kOffBar;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar0 + 8 * (B_FULL + s), 2 * 128);   // a group's 128 threads x (copies landed + stores)
      ptx::mbar_init(bar0 + 8 * (B_EMPTY + s), 1);        // the commit after the step's value MMA
    }
    ptx::mbar_init(bar0 + 8 * B_S, 1);
    ptx::mbar_init(bar0 + 8 * (B_S + 1), 1);
    ptx::mbar_init(bar0 + 8 * B_P, 1);                     // one softmax thread, once the weights are written
    ptx::mbar_init(bar0 + 8 * (B_P + 1), 1);
    ptx::mbar_init(bar0 + 8 * B_NEVER, 1);                 // nothing arrives (failure-path test builds only)
    ptx::mbar_init(bar0 + 8 * B_DRAIN, 1);                 // the score warp's commit when it gives up
    ptx::mbar_init(bar0 + 8 * (B_DRAIN + 1), 1);           // the value warp's
    *abort = 0;
    *bad_flag = 0;
    ptx::fence_mbar_init();
  }
  // both P slots start at zero: the rows of unused head slots (G < 8) stay so
  for (int i = tid; i < 2 * 4096 / 16; i += kThreads) reinterpret_cast<uint4 *>(sm + kOffP)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  if (warp == 0) ptx::tmem_alloc(ptx::smem_addr(tmem_p), kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_p;

  if (warp >= kProdWarp0) {
    const int pwarp = warp - kProdWarp0;
    producer<G>(pr, items, sm, s_base, pwarp / 4, pwarp % 4, lane, abort, bad_flag);
  } else if (warp == kMmaWarp) {
    // Score MMAs. The whole warp walks the steps in lockstep; one elected lane issues.
    StepWalk sw;
    sw.w = blockIdx.x;
    sw.items = items;
    sw.seek(pr);
#ifdef IDX_TEST_STALL
    // Failure-path test builds only: CTA 0's score warp first waits for a barrier
    // nothing ever arrives on, so the wait gives up, raises the abort flag and
    // the CTA leaves without issuing an MMA.
    if (blockIdx.x == 0) ptx::mbar_wait(bar0 + 8 * B_NEVER, 0u, abort, kWaitNs);
#endif
    for (uint32_t j = 0; sw.valid; ++j, sw.next(pr)) {
      // S^T of step j once its stage is full and its S slot's last reader, the
      // softmax of step j - 2, has written its weights
      bool ok = *abort == 0 && ptx::mbar_wait(full_bar(bar0, j), (j / kStages) & 1u, abort, kWaitNs);
      if (ok && j >= 2) ok = ptx::mbar_wait(bar0 + 8 * (B_P + static_cast<int>(j & 1)), ((j - 2) >> 1) & 1u, abort, kWaitNs);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      issue_scores(s_base, tmem, j);
    }
    __syncwarp();
    if (*abort) drain_mmas(bar0 + 8 * B_DRAIN);
  } else if (warp == kMmaWarp + 1) {
    // Value MMAs: O of step j once its weights are written (a second issuing warp, so
    // a step's value MMAs need not wait behind the issue of the next step's scores).
    StepWalk sw;
    sw.w = blockIdx.x;
    sw.items = items;
    sw.seek(pr);
    for (uint32_t j = 0; sw.valid; ++j, sw.next(pr)) {
      const bool ok =
          *abort == 0 && ptx::mbar_wait(bar0 + 8 * (B_P + static_cast<int>(j & 1)), (j >> 1) & 1u, abort, kWaitNs);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      issue_values(s_base, tmem, j, sw.base == 0, 16u * sw.par);   // an item's first step restarts its O slot
    }
    __syncwarp();
    if (*abort) drain_mmas(bar0 + 8 * (B_DRAIN + 1));
  } else {
    constexpr int HPW = (G + 1) / 2;           // head slots a warp serves (with G = 1 the upper warps' slot is unused)
    const int qd = warp & 3, hh = warp >> 2;   // lane quarter; heads HPW hh .. HPW hh + HPW - 1
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    bool ok = true;
    uint32_t j = 0;                            // the CTA's step counter (the launch keeps it below 2^31)
    int item_parity = 0;
    unsigned char *pslot = sm + kOffP;
    const int tok = 32 * qd + lane;
    // this thread's weights p = exp(S - ref) of its heads (token tok) into a P slot,
    // split into bf16 high (rows h) and low (rows 8 + h) parts; their sum in lp
    auto write_weights = [&](unsigned char *pb, const float (&sc)[HPW], const float (&mref)[HPW], float (&lp)[HPW]) {
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        const int h = HPW * hh + i;
        // ex2-based exp: the argument is at most kLazy; relative error a few 1e-7
        const float e = (sc[i] != -INFINITY) ? __expf(sc[i] - mref[i]) : 0.0f;
        lp[i] = e;
        const __nv_bfloat16 ehi = __float2bfloat16_rn(e);
        *reinterpret_cast<__nv_bfloat16 *>(pb + sw128(h, tok, 2048)) = ehi;
        *reinterpret_cast<__nv_bfloat16 *>(pb + sw128(8 + h, tok, 2048)) = __float2bfloat16_rn(e - __bfloat162float(ehi));
      }
    };
    // An item's output waits for its last value MMA; it is written after the next
    // item's first step (or at the next item's end, or the CTA's), so the tensor
    // pipe does not drain at each item's end. O and the sums alternate by item parity.
    bool pend = false, pend_steps = false, pend_fail = false;
    long long pend_out = 0;             // the item's first output element
    uint32_t pend_bar = 0, pend_ph = 0;  // its last step's empty barrier and phase parity
    int pend_par = 0;
    auto flush = [&]() -> bool {
      bool f_ok = true;
      uint32_t ohi[HPW] = {}, olo[HPW] = {};
      if (pend_steps) {   // O is complete once the item's last stage is free again
        f_ok = ptx::mbar_wait(pend_bar, pend_ph, abort, kWaitNs);
        ptx::tc_fence_after();
        if (f_ok) {
          tmem_ldn<HPW>(t_lane + 32 + 16 * pend_par + HPW * hh, ohi);
          tmem_ldn<HPW>(t_lane + 40 + 16 * pend_par + HPW * hh, olo);
          ptx::tmem_wait_ld();
        }
      }
      const float *rs = red + 4 * kGroup * (1 + pend_par);
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        const int h = HPW * hh + i;
        const float L = rs[h] + rs[kGroup + h] + rs[2 * kGroup + h] + rs[3 * kGroup + h];
        const float o = __uint_as_float(ohi[i]) + __uint_as_float(olo[i]);
        if (h < G) pr.out[pend_out + h * kHd + 32 * qd + lane] = L > 0.0f ? o / L : 0.0f;
      }
      ptx::tc_fence_before();   // the reads of O come before the first value MMA of the item after next
      pend = false;
      return f_ok;
    };
    for (uint32_t w = blockIdx.x; w < items && ok; w += gridDim.x, item_parity ^= 1) {
      Item it;
      it.set(pr, w);
      float mref[HPW], lsum[HPW];
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        mref[i] = -INFINITY;
        lsum[i] = 0.0f;
      }
      // one 128-token step of the item (the first one is peeled: after it the previous
      // item's output is written)
      auto step = [&](uint32_t base) {
        const int s = static_cast<int>(j % kStages), b = static_cast<int>(j & 1);
        // the stage's mask (producers' stores) and the step's S^T
        bool w_ok = ptx::mbar_wait(bar0 + 8 * (B_FULL + s), static_cast<uint32_t>((j / kStages) & 1), abort, kWaitNs);
        w_ok = w_ok && ptx::mbar_wait(bar0 + 8 * (B_S + b), static_cast<uint32_t>((j >> 1) & 1), abort, kWaitNs);
        ptx::tc_fence_after();
        const bool valid = (reinterpret_cast<const uint32_t *>(sm + s * kStageBytes + kOffMask)[qd] >> lane) & 1u;
        uint32_t shi[HPW], slo[HPW];
        tmem_ldn<HPW>(t_lane + 16 * b + HPW * hh, shi);
        tmem_ldn<HPW>(t_lane + 16 * b + 8 + HPW * hh, slo);
        ptx::tmem_wait_ld();
        float sc[HPW];
        bool exceed = false;   // a score above its head's reference by more than kLazy
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
          sc[i] = valid ? __uint_as_float(shi[i]) + __uint_as_float(slo[i]) : -INFINITY;
          exceed |= sc[i] > mref[i] + kLazy;   // (any finite score while mref = -inf)
        }
        // Weights against the current references, written as if none moves: the
        // common case needs one barrier a step. P slot b was last read by the value
        // MMA of step j - 2 (another warp issues those: its commit, not this step's
        // S^T, says it is done; the stage's next phase needs weights of step j + 1).
        if (j >= 2) {
          const uint32_t jp = j - 2;
          w_ok = w_ok && ptx::mbar_wait(bar0 + 8 * (B_EMPTY + static_cast<int>(jp % kStages)),
                                        (jp / kStages) & 1u, abort, kWaitNs);
        }
        float lpart[HPW];
        write_weights(pslot + 4096 * b, sc, mref, lpart);
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        if (compute_sync_count(exceed || !w_ok || pend_fail) != 0) {
          // Some reference moves (an item's first step, or a jump): the heads' maxima
          // over the step, then the weights again.
          ok = compute_sync_and(w_ok && !pend_fail);
          if (!ok) return;
#pragma unroll
          for (int i = 0; i < HPW; ++i) {
            const float m = warp_max(sc[i]);
            if (lane == 0) red[qd * kGroup + HPW * hh + i] = m;
          }
          compute_sync_and(true);
          uint32_t rescale = 0;   // bit i: head HPW hh + i's reference moved after an earlier step contributed
          float corr[HPW];
#pragma unroll
          for (int i = 0; i < HPW; ++i) {
            const int h = HPW * hh + i;
            const float tm = fmaxf(fmaxf(red[h], red[kGroup + h]), fmaxf(red[2 * kGroup + h], red[3 * kGroup + h]));
            corr[i] = 1.0f;
            if (tm > mref[i] + kLazy) {
              corr[i] = (mref[i] == -INFINITY) ? 0.0f : __expf(mref[i] - tm);
              if (base > 0) rescale |= 1u << i;
              mref[i] = tm;
              lsum[i] *= corr[i];
            }
          }
          if (rescale) {   // the value MMA of step j - 1 is done once its stage is free again
            const uint32_t jp = j - 1;
            w_ok = ptx::mbar_wait(bar0 + 8 * (B_EMPTY + static_cast<int>(jp % kStages)),
                                  static_cast<uint32_t>((jp / kStages) & 1), abort, kWaitNs);
            ptx::tc_fence_after();
            uint32_t ohi[HPW], olo[HPW];
            const uint32_t oc = t_lane + 32 + 16 * item_parity + HPW * hh;
            tmem_ldn<HPW>(oc, ohi);
            tmem_ldn<HPW>(oc + 8, olo);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < HPW; ++i)
              if ((rescale >> i) & 1u) {
                ohi[i] = __float_as_uint(__uint_as_float(ohi[i]) * corr[i]);
                olo[i] = __float_as_uint(__uint_as_float(olo[i]) * corr[i]);
              }
            tmem_stn<HPW>(oc, ohi);
            tmem_stn<HPW>(oc + 8, olo);
            ptx::tmem_wait_st();
          }
          write_weights(pslot + 4096 * b, sc, mref, lpart);
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before();
          ok = compute_sync_and(w_ok);
          if (!ok) return;
        }
#pragma unroll
        for (int i = 0; i < HPW; ++i) lsum[i] += lpart[i];
        if (tid == 0) ptx::mbar_arrive(bar0 + 8 * (B_P + b));
      };
      uint32_t base = 0;
      if (base < it.n_virt) {
        step(base);
        base += kTok;
        ++j;
        // the previous item's output (its last value MMA went before this step's; the
        // stage's next phase needs weights of a later step, so the wait cannot miss it)
        if (ok && pend) pend_fail = !flush();
      }
      for (; ok && base < it.n_virt; base += kTok, ++j) step(base);
      if (!ok) break;
      if (pend) {   // an item without steps: the previous item's sums need a barrier first
        ok = compute_sync_and(!pend_fail);
        if (!ok) break;
        ok = compute_sync_and(flush());
        if (!ok) break;
      }
      // ---- the item's sums; its output once its last value MMA is done ----
      float *rs = red + 4 * kGroup * (1 + item_parity);
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        float l = lsum[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
        if (lane == 0) rs[qd * kGroup + HPW * hh + i] = l;
      }
      pend = true;
      pend_steps = it.n_virt > 0;
      pend_out = (static_cast<long long>(it.r) * pr.nq + it.kvh * G) * kHd;
      pend_bar = bar0 + 8 * (B_EMPTY + static_cast<int>((j - 1) % kStages));
      pend_ph = static_cast<uint32_t>(((j - 1) / kStages) & 1);
      pend_par = item_parity;
    }
    if (ok && pend) {   // the CTA's last item
      ok = compute_sync_and(!pend_fail);
      if (ok) ok = compute_sync_and(flush());
    }
    if (!ok) *abort = 1;
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (tid == 0 && dev_status) {
    if (*bad_flag) atomicOr(dev_status, IDX_STATUS_BAD_BLOCK);
    if (*abort) atomicOr(dev_status, IDX_STATUS_TIMEOUT);
  }
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool qsa_attn_tc_supported(const float *q, uint32_t nq, uint32_t nkv, uint32_t hd, const void *kc, const void *vc,
                           uint32_t rows, uint32_t first_pos, uint32_t topk, uint32_t ratio, int P,
                           uint32_t block_size) {
  // 1, 2, 4 or 8 query heads per kv head; q is read as float2 pairs, K and V rows by 16-byte copies
  // (their cache rows, P x block_size x nkv of them, are numbered in 31 bits);
  // the steps of all items (at most (topk + 1) ratio tokens an item), the items, positions
  // and token numbers fit the kernel's 32-bit counters
  const unsigned long long tokens = (static_cast<unsigned long long>(topk) + 1) * ratio;
  const unsigned long long steps = static_cast<unsigned long long>(rows) * nkv * (tokens / kTok + 1);
  return hd == kHd && nkv > 0 && (nq == nkv * 8 || nq == nkv * 4 || nq == nkv * 2 || nq == nkv) &&
         steps < (1ull << 31) && tokens < (1ull << 31) &&
         static_cast<unsigned long long>(P) * block_size * nkv < (1ull << 31) &&
         static_cast<unsigned long long>(first_pos) + rows < (1ull << 31) &&
         (reinterpret_cast<uintptr_t>(q) & 7u) == 0 &&
         (reinterpret_cast<uintptr_t>(kc) & 15u) == 0 && (reinterpret_cast<uintptr_t>(vc) & 15u) == 0;
}

cudaError_t launch_qsa_attn_tc(const float *q, const uint16_t *kc, const uint16_t *vc, const int32_t *table,
                               int n_pages, int P, const int32_t *lists, float *out, uint32_t rows, uint32_t first_pos,
                               uint32_t topk, uint32_t ratio, uint32_t block_size, uint32_t nq, uint32_t nkv,
                               float inv_sqrt_d, int32_t *dev_status, cudaStream_t stream) {
  const uint32_t G = nq / nkv;
  void (*kern)(Problem, uint32_t, int32_t *) =
      G == 8 ? qsa_prefill_attn_tc_kernel<8> : G == 4 ? qsa_prefill_attn_tc_kernel<4>
             : G == 2 ? qsa_prefill_attn_tc_kernel<2> : qsa_prefill_attn_tc_kernel<1>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // set on every call: the attribute belongs to the current device's context
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const uint32_t items = rows * nkv;   // below 2^31 (checked with the support)
  const int grid = static_cast<int>(items < static_cast<uint32_t>(sms) ? items : static_cast<uint32_t>(sms));
  const Problem pr{q, kc, vc, table, lists, out, n_pages, P, first_pos, topk, ratio, block_size, nq, nkv,
                   inv_sqrt_d, div_magic(ratio), div_magic(block_size)};
  kern<<<grid, kThreads, kSmemBytes, stream>>>(pr, items, dev_status);
  return cudaGetLastError();
}

}  // namespace idx
