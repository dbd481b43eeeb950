// prefill.cu -- prefill-side sparsification score over the instruction window, for sm_103a.
//
// After a prompt of L tokens, the score of key i in kv head g is the sum, over the window rows
// j in [L - alpha, L) (the instruction tokens) and the G query heads of the group, of the causal
// softmax probability A[j][i] = exp(scale * q_j . k_i - lse_j), i <= j ("How KV Sparsity Achieves
// 1.5x Acceleration for vLLM", section "2. Attention modification": the PyramidKV-style score,
// computed from the forward pass's rowmax and l, whose log-sum-exp is lse_j).
//
// Two kernels, both on warp-level mma.m16n8k16 (bf16 inputs, exact products, fp32 sums):
//  * prefill_score_kernel -- the page's k-outer loop order.  A CTA owns 128 keys of one
//    (sequence, kv head) with their K fragments in registers and streams the window's query
//    columns (column = window row x query head of the group) through a ring of TMA boxes; a key's
//    sum stays in the registers of the lane that holds it, so no sum crosses warps or CTAs.
//    Window rows that lie before the CTA's first key attend none of its keys and are not read
//    (causality), and CTAs past the prompt exit at once.
//  * prefill_lse_kernel -- only when the caller has no lse: the q-outer order.  A CTA owns 128
//    query columns as register fragments and streams the sequence's K blocks up to its last
//    attended key through a TMA ring, keeping a running max (moved lazily) and sum per column.
// Every wait is bounded; bad block ids are skipped and recorded, never dereferenced.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kScoreWarps = 8;
constexpr int kScoreKeys = 32 * kScoreWarps;  // keys per score CTA: two 16-row m-tiles per warp
constexpr int kScoreTiles = kScoreKeys / 16;  // pool blocks per score CTA
constexpr int kQBox = 64 * 128;               // a chunk's d-half box: up to 64 columns x 128 bytes
constexpr int kQSlotBytes = 2 * kQBox;
constexpr int kQOwnSlots = 2;                 // query slots of their own; once the K fragments are in
constexpr int kQSlots = kQOwnSlots + kScoreTiles * 4096 / kQSlotBytes;  // registers, the K tiles' area holds more
constexpr int kLseWarps = 8;
constexpr int kLseMT = 1;                     // 16-column m-tiles per lse warp (two: fewer CTAs and a spill, slower)
constexpr int kLseCols = 16 * kLseMT * kLseWarps;  // query columns per lse CTA
constexpr int kKSlots = 16;                   // K blocks in flight per lse CTA
constexpr float kLseSlack = 8.0f;             // running max moves only when exceeded by this (base 2)
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

template <int D>
__host__ __device__ constexpr int tile_bytes() {
  return 16 * D * 2;
}

// Byte offset of row r, 16-byte chunk c of a bf16 tile written by TMA as boxes of 64 columns
// (128 bytes) with the 128-byte swizzle (chunk XOR row % 8), box b at b * box_stride.
__device__ __forceinline__ uint32_t swz(int r, int c, int box_stride) {
  return (uint32_t)((c >> 3) * box_stride + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); }

// 2^x by the hardware approximation (the PTX ex2 instruction; relative error ~2^-22, results
// below 2^-126 flushed to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// -------------------------------------------------------------------------- score kernel

template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32) prefill_score_kernel(const __grid_constant__ PrefillArgs a) {
  constexpr int KS = D / 16;
  constexpr int TB = tile_bytes<D>();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ktiles = align1024(smem_raw);
  unsigned char* qown = ktiles + kScoreTiles * 4096;  // the K area is sized for d = 128 (as 4 slots)
  uint64_t* bars = reinterpret_cast<uint64_t*>(qown + kQOwnSlots * kQSlotBytes);
  // query slot s: the own slots first, then the K tiles' area once the fragments are loaded
  auto qslot = [&](int slot) -> unsigned char* {
    return slot < kQOwnSlots ? qown + slot * kQSlotBytes : ktiles + (slot - kQOwnSlots) * kQSlotBytes;
  };
  uint64_t* bar_k = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = bars + 1 + kQSlots;
  uint32_t* s_tile_ok = reinterpret_cast<uint32_t*>(bars + 1 + 2 * kQSlots);
  float* lse2 = reinterpret_cast<float*>(s_tile_ok + 4);  // every window column's lse, base 2

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int b = blockIdx.z, g = blockIdx.y;
  const int key0 = blockIdx.x * kScoreKeys;
  const int G = a.G, alpha = a.alpha;

  if (threadIdx.x == 0) {
    mbar_init(bar_k, 1);
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], kScoreWarps);
    }
    fence_mbar_init();
  }
  grid_dependency_wait();  // the lse kernel (or the caller's producer) may still be running
  grid_launch_dependents();

  const int L = a.context_lens[b];
  if (L < 0 || L > a.MB * 16) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
    return;
  }
  if (key0 >= L) return;  // past the prompt
  if (L > a.score_stride && threadIdx.x == 0 && blockIdx.x == 0 && g == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
  // window rows whose position L - alpha + r reaches this CTA's first key
  const int first_row = max(max(0, alpha - L), key0 - (L - alpha));
  const int n_chunks = (alpha - first_row + a.R - 1) / a.R;  // >= 1: position L - 1 >= key0
  const int chunk_bytes = (D / 64) * G * a.R * 128;
  const uint64_t pol_q = l2_policy_evict_last();  // every key block of the sequence reads the window

  int q_issued = 0;  // thread 0: chunks issued so far
  auto issue_q = [&](int i) {
    const int slot = i % kQSlots;
    ++q_issued;
    mbar_arrive_expect_tx(&q_full[slot], (uint32_t)chunk_bytes);
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx)
      tma_load_3d(qslot(slot) + bx * kQBox, &a.tmap_q, bx * 64, g * G, b * alpha + first_row + i * a.R,
                  &q_full[slot], pol_q);
  };

  __syncthreads();  // barriers initialised
  if (threadIdx.x == 0) {
    const uint64_t pol_k = l2_policy_evict_first();
    uint32_t ok = 0, bytes = 0;
    int phys[kScoreTiles];
#pragma unroll
    for (int p = 0; p < kScoreTiles; ++p) {
      const int u = key0 / 16 + p;
      phys[p] = -1;
      if (u * 16 < L) {
        const int pb = a.block_tables[(size_t)b * a.MB + u];
        if (pb >= 0 && pb < a.NB) {
          phys[p] = pb;
          ok |= 1u << p;
          bytes += TB;
        } else {
          record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
        }
      }
    }
    *s_tile_ok = ok;
    mbar_arrive_expect_tx(bar_k, bytes);
#pragma unroll
    for (int p = 0; p < kScoreTiles; ++p) {
      if (!((ok >> p) & 1u)) continue;
      const int y = (phys[p] * a.Hkv + g) * 16;  // host checks NB*Hkv*16 < 2^31
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx) tma_load_2d(ktiles + p * TB + bx * 2048, &a.tmap_k, bx * 64, y, bar_k, pol_k);
    }
    for (int i = 0; i < kQOwnSlots && i < n_chunks; ++i) issue_q(i);
  }
  // stage every window column's lse in base 2 (column c = window row c / G, head g G + c % G)
  for (int c = threadIdx.x; c < alpha * G; c += blockDim.x) {
    const int r = c / G, hi = c - r * G;
    lse2[c] = a.lse[((size_t)b * a.Hq + (size_t)g * G + hi) * alpha + r] * kLog2eF;
  }
  __syncthreads();

  bool aborted = false;
  if (!__all_sync(kFullMask, mbar_wait_bounded(bar_k, 0, a.timeout_ns))) {
    if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
    aborted = true;
  }
  // this warp's keys: two m-tiles (pool blocks 2 warp, 2 warp + 1), rows gq and gq + 8 of each
  const uint32_t tiles_ok = *s_tile_ok;
  uint32_t af[2][KS][4];
  int key[2][2];
  bool kval[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int p = 2 * warp + mt;
    const uint32_t tb = smem_u32(ktiles + p * TB);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) ldsm_x4(tb + swz(lane & 15, 2 * ks + (lane >> 4), 2048), af[mt][ks]);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      key[mt][rr] = key0 + p * 16 + gq + 8 * rr;
      kval[mt][rr] = !aborted && ((tiles_ok >> p) & 1u) && key[mt][rr] < L;
    }
    // rows of invalid keys (past the prompt, a skipped block) become zeros, so their logits are
    // finite and a 0 factor removes them: af[.][.][0], [2] hold row gq, [1], [3] row gq + 8
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (!kval[mt][0]) af[mt][ks][0] = af[mt][ks][2] = 0u;
      if (!kval[mt][1]) af[mt][ks][1] = af[mt][ks][3] = 0u;
    }
  }
  float kf[2][2];  // 1 for a valid key, 0 otherwise
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) kf[mt][rr] = kval[mt][rr] ? 1.f : 0.f;
  // every warp has its fragments: the K tiles' area now takes query chunks
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0 && !aborted)
    for (int i = kQOwnSlots; i < kQSlots && i < n_chunks; ++i) issue_q(i);
  const int key_last = min(key0 + kScoreKeys, L) - 1;
  const float sl2 = a.scale_log2;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};

  int i = 0;
  for (; i < n_chunks && !aborted; ++i) {
    const int slot = i % kQSlots;
    const uint32_t parity = (uint32_t)(i / kQSlots) & 1u;
    if (!__all_sync(kFullMask, mbar_wait_bounded(&q_full[slot], parity, a.timeout_ns))) {
      if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    const int rs = first_row + i * a.R;
    const int ncols = min(a.R, alpha - rs) * G;
    const int jbase = L - alpha + rs;           // position of the chunk's first row
    const bool all_attended = key_last <= jbase;  // every key here precedes every row
    const uint32_t qbase = smem_u32(qslot(slot));
    for (int n8 = 0; n8 < ncols; n8 += 8) {
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
        uint32_t bq[4];
        ldsm_x4(qbase + swz(n8 + (lane & 7), 4 * kp + (lane >> 3), kQBox), bq);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_bf16_m16n8k16(c[mt], af[mt][2 * kp], bq[0], bq[1]);
          mma_bf16_m16n8k16(c[mt], af[mt][2 * kp + 1], bq[2], bq[3]);
        }
      }
      // this lane's columns: n8 + 2tq and n8 + 2tq + 1 of the chunk
      const int cc0 = n8 + 2 * tq, cc1 = cc0 + 1;
      if (all_attended && n8 + 8 <= ncols) {
        // every key of the CTA precedes every row of the chunk: no causal or column masks
        const float l0 = lse2[rs * G + cc0], l1 = lse2[rs * G + cc1];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float e = ex2(fmaf(c[mt][2 * rr], sl2, -l0)) + ex2(fmaf(c[mt][2 * rr + 1], sl2, -l1));
            acc[mt][rr] = fmaf(kf[mt][rr], e, acc[mt][rr]);
          }
      } else {
        const bool cv0 = cc0 < ncols, cv1 = cc1 < ncols;
        const float l0 = cv0 ? lse2[rs * G + cc0] : 0.f;
        const float l1 = cv1 ? lse2[rs * G + cc1] : 0.f;
        const int j0 = jbase + cc0 / G, j1 = jbase + cc1 / G;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int k = key[mt][rr];
            const bool a0 = kval[mt][rr] && cv0 && k <= j0;
            const bool a1 = kval[mt][rr] && cv1 && k <= j1;
            const float e0 = ex2(fmaf(c[mt][2 * rr], sl2, -l0));
            const float e1 = ex2(fmaf(c[mt][2 * rr + 1], sl2, -l1));
            acc[mt][rr] += (a0 ? e0 : 0.f) + (a1 ? e1 : 0.f);
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[slot]);
    if (threadIdx.x == 0 && i + kQSlots < n_chunks) {
      if (!mbar_wait_bounded(&q_empty[slot], parity, a.timeout_ns)) {
        record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
      } else {
        fence_proxy_async_smem();
        issue_q(i + kQSlots);
      }
    }
  }
  if (threadIdx.x == 0) {  // let every copy this thread issued land before the CTA exits
    for (int k = i; k < q_issued; ++k)
      (void)mbar_wait_bounded(&q_full[k % kQSlots], (uint32_t)(k / kQSlots) & 1u, a.timeout_ns);
    (void)mbar_wait_bounded(bar_k, 0, a.timeout_ns);
  }
  if (aborted) return;
  // a key's sum is spread over the 4 lanes of its row group
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float v = acc[mt][rr];
      v += __shfl_xor_sync(kFullMask, v, 1);
      v += __shfl_xor_sync(kFullMask, v, 2);
      const int k = key[mt][rr];
      if (tq == 0 && kval[mt][rr] && k < a.score_stride) {
        float* dst = a.scores + ((size_t)b * a.Hkv + g) * a.score_stride + k;
        *dst += v;
      }
    }
}

// ------------------------------------------------------------ score kernel on tcgen05 (UMMA)
//
// The same k-outer score, with the contraction on the 5th-generation tensor cores: a CTA (one
// per SM) owns 256 keys of one (sequence, kv head) as two 128-key halves; each half's K tile is
// an A operand (128 keys x 128 d, K-major, 128-byte swizzle, as TMA writes it), each chunk of 128
// window columns the B operand both halves share (so each CTA reads the window once per 256 keys),
// and S^T = K Q^T (128 x 128 fp32 per half) accumulates in tensor memory over 8 k-steps of 16.
// Roles: warp 16 issues the TMA copies, one thread of warp 17 issues the MMAs, warps 0-15 read
// the accumulators (warp w reads TMEM lanes 32 (w % 4) .. + 31 of key half (w / 4) % 2, one key per
// thread, and column half w / 8) and add each probability to the thread's key sum; the column
// halves' sums meet in shared memory.  Two accumulators per key half (all 512 TMEM columns) let
// the MMAs of chunk i + 1 run while chunk i is read.  d = 128 and G a power of two (so a chunk is
// whole window rows).
constexpr int kTcKH = PKV_TC_KH;               // 128-key halves per CTA
constexpr int kTcKeys = 128 * kTcKH;
constexpr int kTcCols = PKV_TC_COLS;           // window columns per chunk (the MMA's N; 64 or 128)
constexpr int kTcHalf = 128 * 128;             // one d-half of a 128-key A operand: 128 rows x 128 B
constexpr int kTcQHalf = kTcCols * 128;        // one d-half of a query chunk
constexpr int kTcQSlots = PKV_TC_QSLOTS;       // query chunks in flight
constexpr int kTcAcc = PKV_TC_ACC;             // accumulators per key half in tensor memory
constexpr int kTcReaders = 8 * kTcKH;          // accumulator-reading warps: lane group x key half x column half
constexpr int kTcThreads = 32 * (kTcReaders + 2);
constexpr uint32_t kTcTmemUsed = kTcAcc * kTcKH * kTcCols;
constexpr uint32_t kTcTmemCols = kTcTmemUsed <= 32 ? 32 : kTcTmemUsed <= 64 ? 64 : kTcTmemUsed <= 128 ? 128
                                 : kTcTmemUsed <= 256 ? 256 : 512;  // allocations are powers of two
static_assert(kTcTmemUsed <= 512 && (kTcCols == 64 || kTcCols == 128), "tensor memory / chunk shape");
constexpr int kTcMaxColumns = 8192;            // alpha * G bound of this kernel (its lse copy in shared memory)

__global__ void __launch_bounds__(kTcThreads, PKV_TC_MINB) prefill_score_tc_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sa = align1024(smem_raw);              // A: 2 d-halves x kTcKH x 16 KiB
  unsigned char* sq = sa + 2 * kTcKH * kTcHalf;         // B slots: kTcQSlots x 2 d-halves x kTcQHalf
  uint64_t* bars = reinterpret_cast<uint64_t*>(sq + kTcQSlots * 2 * kTcQHalf);
  uint64_t* k_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + kTcQSlots;
  uint64_t* acc_full = q_empty + kTcQSlots;
  uint64_t* acc_empty = acc_full + kTcAcc;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + kTcAcc);
  uint32_t* s_tiles_ok = s_tmem + 1;
  float* s_half = reinterpret_cast<float*>(s_tmem + 4);  // the second column half's key sums
  // minus the lse (base 2) of the window columns from the CTA's first row; 16-byte aligned
  float* nlse2 = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(s_half + kTcKeys) + 15) & ~uintptr_t(15));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, g = blockIdx.y;
  const int key0 = blockIdx.x * kTcKeys;
  const int G = a.G, alpha = a.alpha;
  const int rows_per_chunk = kTcCols / G;

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < kTcQSlots; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < kTcAcc; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kTcReaders);
    }
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();

  const int L = a.context_lens[b];
  if (L < 0 || L > a.MB * 16) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
    return;
  }
  if (key0 >= L) return;
  if (L > a.score_stride && threadIdx.x == 0 && blockIdx.x == 0 && g == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
  const int first_row = max(max(0, alpha - L), key0 - (L - alpha));
  const int n_chunks = (alpha - first_row + rows_per_chunk - 1) / rows_per_chunk;

  if (warp == 0) {  // tensor memory for the two accumulators
    tmem_alloc(s_tmem, kTcTmemCols);
    tmem_relinquish();
  }
  // minus the lse of the columns from the first row on, chunk-major (chunk i's column c at
  // i * kTcCols + c), so the logit FMA adds it
  for (int k = threadIdx.x; k < (alpha - first_row) * G; k += blockDim.x) {
    const int c = first_row * G + k;
    const int r = c / G, hi = c - r * G;
    nlse2[k] = -a.lse[((size_t)b * a.Hq + (size_t)g * G + hi) * alpha + r] * kLog2eF;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool aborted = false;
  const int lg = warp & 3, kh = (warp >> 2) & (kTcKH - 1), ch = warp / (4 * kTcKH);  // readers
  const int row = 128 * kh + 32 * lg + lane;  // key row of the CTA (TMEM lane 32 lg + lane of half kh)
  const int key = key0 + row;
  bool kval = false;
  float sum = 0.f;

  if (warp == kTcReaders) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_k = l2_policy_evict_first(), pol_q = l2_policy_evict_last();
      uint32_t ok = 0, bytes = 0;
      int phys[kTcKeys / 16];
#pragma unroll
      for (int p = 0; p < kTcKeys / 16; ++p) {
        const int u = key0 / 16 + p;
        phys[p] = -1;
        if (u * 16 < L) {
          const int pb = a.block_tables[(size_t)b * a.MB + u];
          if (pb >= 0 && pb < a.NB) {
            phys[p] = pb;
            ok |= 1u << p;
            bytes += 2 * 2048;
          } else {
            record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
          }
        }
      }
      *s_tiles_ok = ok;
      mbar_arrive_expect_tx(k_full, bytes);
#pragma unroll
      for (int p = 0; p < kTcKeys / 16; ++p) {
        if (!((ok >> p) & 1u)) continue;
        const int y = (phys[p] * a.Hkv + g) * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_2d(sa + h * kTcKH * kTcHalf + p * 2048, &a.tmap_k, h * 64, y, k_full, pol_k);
      }
      int issued = 0;
      for (int i = 0; i < n_chunks; ++i) {
        const int s = i % kTcQSlots;
        if (i >= kTcQSlots && !mbar_wait_bounded(&q_empty[s], (uint32_t)((i / kTcQSlots) - 1) & 1u, a.timeout_ns)) {
          record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
          break;
        }
        const int rs = first_row + i * rows_per_chunk;
        mbar_arrive_expect_tx(&q_full[s], 2 * kTcQHalf);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < kTcCols / 64; ++j)
            tma_load_3d(sq + (s * 2 + h) * kTcQHalf + j * 8192, &a.tmap_q, h * 64, g * G,
                        b * alpha + rs + j * (64 / G), &q_full[s], pol_q);
        ++issued;
      }
      // every copy lands before the CTA may exit
      (void)mbar_wait_bounded(k_full, 0, a.timeout_ns);
      for (int i = max(0, issued - kTcQSlots); i < issued; ++i)
        (void)mbar_wait_bounded(&q_full[i % kTcQSlots], (uint32_t)(i / kTcQSlots) & 1u, a.timeout_ns);
    }
  } else if (warp == kTcReaders + 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, kTcCols);
      int done = 0;
      if (mbar_wait_bounded(k_full, 0, a.timeout_ns)) {
        const uint32_t a0 = smem_u32(sa);
        for (int i = 0; i < n_chunks; ++i) {
          const int s = i % kTcQSlots, acc = i % kTcAcc;
          if (!mbar_wait_bounded(&q_full[s], (uint32_t)(i / kTcQSlots) & 1u, a.timeout_ns)) break;
          if (i >= kTcAcc && !mbar_wait_bounded(&acc_empty[acc], (uint32_t)((i / kTcAcc) - 1) & 1u, a.timeout_ns))
            break;
          tc_fence_after();
          const uint32_t b0 = smem_u32(sq + s * 2 * kTcQHalf);
#pragma unroll
          for (int kh = 0; kh < kTcKH; ++kh)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t aoff = (uint32_t)(((k >> 2) * kTcKH + kh) * kTcHalf + (k & 3) * 32);
              const uint32_t boff = (uint32_t)((k >> 2) * kTcQHalf + (k & 3) * 32);
              umma_bf16(tmem + (acc * kTcKH + kh) * kTcCols, umma_desc_sw128(a0 + aoff), umma_desc_sw128(b0 + boff),
                        idesc, k > 0);
            }
          umma_commit(&q_empty[s]);
          umma_commit(&acc_full[acc]);
          ++done;
        }
      } else {
        record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      }
      if (done > 0)  // the last MMAs complete before the CTA may release tensor memory
        (void)mbar_wait_bounded(&acc_full[(done - 1) % kTcAcc], (uint32_t)((done - 1) / kTcAcc) & 1u, a.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------------- accumulator readers
    kval = key < L;
    const float sl2 = a.scale_log2;
    const int key_last = min(key0 + kTcKeys, L) - 1;
    const int log2g = 31 - __clz(G);
    if (!__all_sync(kFullMask, mbar_wait_bounded(k_full, 0, a.timeout_ns))) {
      if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      aborted = true;
    }
    kval = kval && ((*s_tiles_ok >> (row >> 4)) & 1u);
    for (int i = 0; i < n_chunks && !aborted; ++i) {
      const int acc = i % kTcAcc;
      if (!__all_sync(kFullMask, mbar_wait_bounded(&acc_full[acc], (uint32_t)(i / kTcAcc) & 1u, a.timeout_ns))) {
        if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t t = tmem + ((uint32_t)(32 * lg) << 16) + (acc * kTcKH + kh) * kTcCols;
      const int rs = first_row + i * rows_per_chunk;
      const int ncols = min(rows_per_chunk, alpha - rs) * G;
      const int jbase = L - alpha + rs;
      const bool fast = ncols == kTcCols && key_last <= jbase;  // whole chunk, every key before every row
      const float* l2c = nlse2 + i * kTcCols;
#pragma unroll 1
      for (int q = ch * (kTcCols / 64); q < (ch + 1) * (kTcCols / 64); ++q) {  // this warp's half, 32 at a time
        float v[32];
        tmem_ld_x32(t + 32 * q, v);
        tmem_wait_ld();
        if (kval) {
          if (fast) {  // packed fp32 pairs: one FMA and one add per two probabilities
            const uint64_t s2 = pack2(sl2, sl2);
            uint64_t acc2 = pack2(0.f, 0.f);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 l = *reinterpret_cast<const float4*>(l2c + 32 * q + 4 * c4);
              const float2 x01 = unpack2(ffma2(pack2(v[4 * c4], v[4 * c4 + 1]), s2, pack2(l.x, l.y)));
              const float2 x23 = unpack2(ffma2(pack2(v[4 * c4 + 2], v[4 * c4 + 3]), s2, pack2(l.z, l.w)));
              acc2 = fadd2(acc2, pack2(ex2(x01.x), ex2(x01.y)));
              acc2 = fadd2(acc2, pack2(ex2(x23.x), ex2(x23.y)));
            }
            const float2 a2 = unpack2(acc2);
            sum += a2.x + a2.y;
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int cc = 32 * q + c;
              if (cc < ncols && key <= jbase + (cc >> log2g)) sum += ex2(fmaf(v[c], sl2, l2c[cc]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
    if (aborted) kval = false;
    if (ch == 1) s_half[row] = kval ? sum : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  if (ch == 0 && warp < kTcReaders && kval && key < a.score_stride)
    a.scores[((size_t)b * a.Hkv + g) * a.score_stride + key] += sum + s_half[row];
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ---------------------------------------------------------------- lse kernel on tcgen05 (UMMA)
//
// The window rows' log-sum-exps when the caller has none: the q-outer order on tcgen05.  A CTA
// owns 128 window columns of one (sequence, kv head) as the A operand (TMA boxes of the window's
// queries, K-major, 128-byte swizzle); the sequence's K streams as B operands in chunks of 128
// keys (8 pool blocks) through a ring, up to the CTA's last attended key; S = Q K^T (128 x 128
// fp32) accumulates in tensor memory.  Warp 8 issues the TMA copies, one thread of warp 9 the
// MMAs, warps 0-7 read the accumulators (warp w: TMEM lanes 32 (w % 4) .., one column per
// thread, key half w / 4 of each chunk) and keep a running max (moved lazily) and sum; the two
// halves merge in shared memory.  d = 128 and G a power of two.
constexpr int kLtKSlots = 2;
constexpr int kLtThreads = 32 * 10;

__global__ void __launch_bounds__(kLtThreads, 2) prefill_lse_tc_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sa = align1024(smem_raw);                // A: 2 d-halves x 128 columns x 128 B
  unsigned char* sk = sa + 2 * kTcHalf;                   // B slots: kLtKSlots x 2 d-halves x 128 keys x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sk + kLtKSlots * 2 * kTcHalf);
  uint64_t* a_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kLtKSlots;
  uint64_t* acc_full = k_empty + kLtKSlots;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + 2);
  float2* s_half = reinterpret_cast<float2*>(s_tmem + 4); // the second key half's (m, l) per column
  int32_t* s_bt = reinterpret_cast<int32_t*>(s_half + 128);  // the sequence's block ids

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, g = blockIdx.y;
  const int cbase = blockIdx.x * 128;
  const int G = a.G, alpha = a.alpha;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < kLtKSlots; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 8);
    }
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();

  const int L = a.context_lens[b];
  if (L < 0 || L > a.MB * 16) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
    return;
  }
  const int ncol = alpha * G;
  const int c_lo = max(0, alpha - L) * G;  // columns of rows before position 0 have no keys
  if (cbase >= ncol) return;
  auto lse_at = [&](int c) -> float* {
    return a.lse + ((size_t)b * a.Hq + (size_t)g * G + (c & (G - 1))) * alpha + c / G;
  };
  for (int c = cbase + (int)threadIdx.x; c < min(cbase + 128, c_lo); c += blockDim.x) *lse_at(c) = -INFINITY;
  if (cbase + 128 <= c_lo) return;
  const int c_last = min(cbase + 128, ncol) - 1;
  const int j_last = L - alpha + c_last / G;             // the CTA's last attended key
  const int n_chunks = j_last / 128 + 1;
  const int nblk = j_last / 16 + 1;
  for (int u = threadIdx.x; u < nblk; u += blockDim.x) s_bt[u] = a.block_tables[(size_t)b * a.MB + u];
  if (warp == 0) {
    tmem_alloc(s_tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  bool aborted = false;
  const int lg = warp & 3, kh = warp >> 2;  // readers: TMEM lane group, key half of each chunk
  const int row = 32 * lg + lane;           // this thread's column of the CTA
  const int col = cbase + row;
  float m = -INFINITY, l = 0.f;             // running max (base 2) and sum over this thread's keys

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first(), pol_k = l2_policy_evict_last();
      mbar_arrive_expect_tx(a_full, 2 * kTcHalf);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(sa + h * kTcHalf + j * 8192, &a.tmap_q, h * 64, g * G, b * alpha + cbase / G + j * (64 / G),
                      a_full, pol_q);
      int issued = 0;
      for (int i = 0; i < n_chunks; ++i) {
        const int s = i % kLtKSlots;
        if (i >= kLtKSlots && !mbar_wait_bounded(&k_empty[s], (uint32_t)((i / kLtKSlots) - 1) & 1u, a.timeout_ns)) {
          record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
          break;
        }
        uint32_t ok = 0, bytes = 0;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int u = 8 * i + p;
          if (u >= nblk) continue;
          const int phys = s_bt[u];
          if (phys >= 0 && phys < a.NB) {
            ok |= 1u << p;
            bytes += 2 * 2048;
          } else {
            record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
          }
        }
        mbar_arrive_expect_tx(&k_full[s], bytes);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          if (!((ok >> p) & 1u)) continue;
          const int y = (s_bt[8 * i + p] * a.Hkv + g) * 16;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sk + (s * 2 + h) * kTcHalf + p * 2048, &a.tmap_k, h * 64, y, &k_full[s], pol_k);
        }
        ++issued;
      }
      // every copy lands before the CTA may exit
      (void)mbar_wait_bounded(a_full, 0, a.timeout_ns);
      for (int i = max(0, issued - kLtKSlots); i < issued; ++i)
        (void)mbar_wait_bounded(&k_full[i % kLtKSlots], (uint32_t)(i / kLtKSlots) & 1u, a.timeout_ns);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, 128);
      int done = 0;
      if (mbar_wait_bounded(a_full, 0, a.timeout_ns)) {
        const uint32_t a0 = smem_u32(sa);
        for (int i = 0; i < n_chunks; ++i) {
          const int s = i % kLtKSlots, acc = i & 1;
          if (!mbar_wait_bounded(&k_full[s], (uint32_t)(i / kLtKSlots) & 1u, a.timeout_ns)) break;
          if (i >= 2 && !mbar_wait_bounded(&acc_empty[acc], (uint32_t)((i >> 1) - 1) & 1u, a.timeout_ns)) break;
          tc_fence_after();
          const uint32_t b0 = smem_u32(sk + s * 2 * kTcHalf);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (uint32_t)((k >> 2) * kTcHalf + (k & 3) * 32);
            umma_bf16(tmem + acc * 128, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, k > 0);
          }
          umma_commit(&k_empty[s]);
          umma_commit(&acc_full[acc]);
          ++done;
        }
      } else {
        record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      }
      if (done > 0)  // the last MMAs complete before the CTA may release tensor memory
        (void)mbar_wait_bounded(&acc_full[(done - 1) & 1], (uint32_t)((done - 1) >> 1) & 1u, a.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------------- accumulator readers
    const float sl2 = a.scale_log2;
    const int j = L - alpha + col / G;                               // this column's position
    const int j_min = L - alpha + max(cbase, c_lo) / G;              // the CTA's first valid position
    for (int i = 0; i < n_chunks && !aborted; ++i) {
      const int acc = i & 1;
      if (!__all_sync(kFullMask, mbar_wait_bounded(&acc_full[acc], (uint32_t)(i >> 1) & 1u, a.timeout_ns))) {
        if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t t = tmem + ((uint32_t)(32 * lg) << 16) + acc * 128;
#pragma unroll 1
      for (int q = 2 * kh; q < 2 * kh + 2; ++q) {  // this warp's 64 keys, 32 at a time
        const int k0 = 128 * i + 32 * q;
        float v[32];
        tmem_ld_x32(t + 32 * q, v);
        tmem_wait_ld();
        const int u0 = k0 >> 4;
        const bool blocks_ok = u0 + 1 < nblk && s_bt[u0] >= 0 && s_bt[u0] < a.NB && s_bt[u0 + 1] >= 0 &&
                               s_bt[u0 + 1] < a.NB;
        if (!(blocks_ok && k0 + 31 <= j_min)) {  // near the diagonal or a skipped block: mask keys
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int k = k0 + c, u = k >> 4;
            const bool kv = k <= j && u < nblk && s_bt[u] >= 0 && s_bt[u] < a.NB;
            v[c] = kv ? v[c] : -INFINITY;
          }
        }
        float mx = v[0];
#pragma unroll
        for (int c = 1; c < 32; ++c) mx = fmaxf(mx, v[c]);
        mx *= sl2;  // sl2 > 0 keeps the order
        if (mx > m + kLseSlack) {
          l *= ex2(m - mx);
          m = mx;
        }
        if (m != -INFINITY) {  // packed fp32 pairs: one FMA and one add per two terms
          const uint64_t s2 = pack2(sl2, sl2), nm2 = pack2(-m, -m);
          uint64_t e2 = pack2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 x = unpack2(ffma2(pack2(v[c], v[c + 1]), s2, nm2));
            e2 = fadd2(e2, pack2(ex2(x.x), ex2(x.y)));
          }
          const float2 e = unpack2(e2);
          l += e.x + e.y;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
    if (kh == 1) s_half[row] = make_float2(m, l);
  }
  tc_fence_before();
  __syncthreads();
  if (warp < 4 && !aborted && col >= c_lo && col < ncol) {
    const float2 o = s_half[row];
    const float M = fmaxf(m, o.x);
    const float lt = (m == -INFINITY ? 0.f : l * exp2f(m - M)) + (o.x == -INFINITY ? 0.f : o.y * exp2f(o.x - M));
    *lse_at(col) = lt > 0.f ? (M + log2f(lt)) * kLn2F : -INFINITY;
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------- lse kernel

template <int D>
__global__ void __launch_bounds__(kLseWarps * 32) prefill_lse_kernel(const __grid_constant__ PrefillArgs a) {
  constexpr int KS = D / 16;
  constexpr int TB = tile_bytes<D>();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ktiles = align1024(smem_raw);
  uint64_t* k_full = reinterpret_cast<uint64_t*>(ktiles + kKSlots * TB);
  uint64_t* k_empty = k_full + kKSlots;
  uint32_t* s_ok = reinterpret_cast<uint32_t*>(k_empty + kKSlots);
  int32_t* s_bt = reinterpret_cast<int32_t*>(s_ok + kKSlots);  // the sequence's block ids, staged once

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int b = blockIdx.z, g = blockIdx.y;
  const int cbase = blockIdx.x * kLseCols;
  const int G = a.G, alpha = a.alpha;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], kLseWarps);
    }
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();

  const int L = a.context_lens[b];
  if (L < 0 || L > a.MB * 16) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
    return;
  }
  const int ncol = alpha * G;
  const int c_lo = max(0, alpha - L) * G;  // columns of rows before position 0 have no keys
  if (cbase >= ncol) return;
  auto lse_at = [&](int c) -> float* {
    return a.lse + ((size_t)b * a.Hq + (size_t)g * G + c % G) * alpha + c / G;
  };
  for (int c = cbase + (int)threadIdx.x; c < min(cbase + kLseCols, c_lo); c += blockDim.x) *lse_at(c) = -INFINITY;
  if (cbase + kLseCols <= c_lo) return;
  const int c_last = min(cbase + kLseCols, ncol) - 1;
  const int nblk = (L - alpha + c_last / G) / 16 + 1;  // blocks up to the CTA's last attended key

  int k_issued = 0;  // thread 0: blocks issued so far
  auto issue_k = [&](int u) {
    const int slot = u % kKSlots;
    ++k_issued;
    const int phys = s_bt[u];
    if (phys >= 0 && phys < a.NB) {
      s_ok[slot] = 1u;
      mbar_arrive_expect_tx(&k_full[slot], TB);
      const int y = (phys * a.Hkv + g) * 16;
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx)
        tma_load_2d(ktiles + slot * TB + bx * 2048, &a.tmap_k, bx * 64, y, &k_full[slot], l2_policy_evict_last());
    } else {
      record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
      s_ok[slot] = 0u;
      mbar_arrive_expect_tx(&k_full[slot], 0);
    }
  };
  for (int u = threadIdx.x; u < nblk; u += blockDim.x) s_bt[u] = a.block_tables[(size_t)b * a.MB + u];
  __syncthreads();  // barriers initialised, block ids staged
  if (threadIdx.x == 0)
    for (int u = 0; u < kKSlots && u < nblk; ++u) issue_k(u);

  // this warp's 16 * kLseMT columns as A operands: m-tile mt, fragment row gq + 8 rr is column
  // cbase + warp * 16 kLseMT + 16 mt + gq + 8 rr; invalid columns are zeros
  int col[kLseMT][2], jpos[kLseMT][2];
  bool cval[kLseMT][2];
  uint32_t aq[kLseMT][KS][4];
#pragma unroll
  for (int mt = 0; mt < kLseMT; ++mt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int c = cbase + warp * 16 * kLseMT + 16 * mt + gq + 8 * rr;
      col[mt][rr] = c;
      cval[mt][rr] = c >= c_lo && c < ncol;
      jpos[mt][rr] = L - alpha + c / G;  // the row's position
      const __nv_bfloat16* qr = a.q_win + (((size_t)b * alpha + c / G) * a.Hq + (size_t)g * G + c % G) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        aq[mt][ks][rr] = cval[mt][rr] ? ld_u32(qr + 16 * ks + 2 * tq) : 0u;
        aq[mt][ks][2 + rr] = cval[mt][rr] ? ld_u32(qr + 16 * ks + 8 + 2 * tq) : 0u;
      }
    }
  // the smallest position among the warp's columns (invalid columns count as the window start)
  const int j_warp = L - alpha + max(cbase + warp * 16 * kLseMT, c_lo) / G;
  const float sl2 = a.scale_log2;
  float m[kLseMT][2], l[kLseMT][2];  // this lane's share of each row: running max (base 2), sum
#pragma unroll
  for (int mt = 0; mt < kLseMT; ++mt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      m[mt][rr] = -INFINITY;
      l[mt][rr] = 0.f;
    }

  bool aborted = false;
  int u = 0;
  for (; u < nblk; ++u) {
    const int slot = u % kKSlots;
    const uint32_t parity = (uint32_t)(u / kKSlots) & 1u;
    if (!__all_sync(kFullMask, mbar_wait_bounded(&k_full[slot], parity, a.timeout_ns))) {
      if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    if (s_ok[slot]) {
      const uint32_t tb = smem_u32(ktiles + slot * TB);
      float sc[kLseMT][2][4] = {};
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          uint32_t bk[4];
          ldsm_x4(tb + swz(8 * n + (lane & 7), 4 * kp + (lane >> 3), 2048), bk);
#pragma unroll
          for (int mt = 0; mt < kLseMT; ++mt) {
            mma_bf16_m16n8k16(sc[mt][n], aq[mt][2 * kp], bk[0], bk[1]);
            mma_bf16_m16n8k16(sc[mt][n], aq[mt][2 * kp + 1], bk[2], bk[3]);
          }
        }
      }
      // sc[mt][n] = (row gq, key 8n + 2tq), (gq, +1), (gq + 8, 8n + 2tq), (gq + 8, +1) of this block
      const bool unmasked = u * 16 + 15 <= j_warp;  // the block precedes every row of this warp
#pragma unroll
      for (int mt = 0; mt < kLseMT; ++mt)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          float x[4];
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int k = u * 16 + 8 * n + 2 * tq + e;  // causal: k <= j (also < L, as j < L)
              x[2 * n + e] = (unmasked || k <= jpos[mt][rr]) ? sc[mt][n][2 * rr + e] : -INFINITY;
            }
          // unscaled logits: sl2 > 0 keeps the order, so the max scales after
          const float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])) * sl2;
          float& mr = m[mt][rr];
          float& lr = l[mt][rr];
          if (mx > mr + kLseSlack) {
            lr *= ex2(mr - mx);
            mr = mx;
          }
          if (mr != -INFINITY)
            lr += ex2(fmaf(x[0], sl2, -mr)) + ex2(fmaf(x[1], sl2, -mr)) + ex2(fmaf(x[2], sl2, -mr)) +
                  ex2(fmaf(x[3], sl2, -mr));
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&k_empty[slot]);
    if (threadIdx.x == 0 && u + kKSlots < nblk) {
      if (!mbar_wait_bounded(&k_empty[slot], parity, a.timeout_ns)) {
        record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
      } else {
        fence_proxy_async_smem();
        issue_k(u + kKSlots);
      }
    }
  }
  if (threadIdx.x == 0) {  // let every copy this thread issued land before the CTA exits
    for (int k = u; k < k_issued; ++k)
      (void)mbar_wait_bounded(&k_full[k % kKSlots], (uint32_t)(k / kKSlots) & 1u, a.timeout_ns);
  }
  if (aborted) return;
  // combine the 4 lanes of each row: (m, l) pairs under a common max
#pragma unroll
  for (int mt = 0; mt < kLseMT; ++mt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float mr = m[mt][rr], lr = l[mt][rr];
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const float m2 = __shfl_xor_sync(kFullMask, mr, o), l2 = __shfl_xor_sync(kFullMask, lr, o);
        const float M = fmaxf(mr, m2);
        lr = (mr == -INFINITY ? 0.f : lr * exp2f(mr - M)) + (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - M));
        mr = M;
      }
      if (tq == 0 && cval[mt][rr]) *lse_at(col[mt][rr]) = lr > 0.f ? (mr + log2f(lr)) * kLn2F : -INFINITY;
    }
}

}  // namespace

size_t prefill_score_smem_bytes(int head_dim, int alpha, int group) {
  (void)head_dim;  // the K tiles' area is sized for d = 128 either way (it doubles as query slots)
  return 1024 + kScoreTiles * 4096 + kQOwnSlots * (size_t)kQSlotBytes + sizeof(uint64_t) * (1 + 2 * kQSlots) + 16 +
         sizeof(float) * (size_t)alpha * group;
}

size_t prefill_score_tc_smem_bytes(int alpha, int group) {
  return 1024 + 2 * kTcKH * kTcHalf + kTcQSlots * 2 * kTcQHalf + sizeof(uint64_t) * (1 + 2 * kTcQSlots + 2 * kTcAcc) +
         16 + sizeof(float) * kTcKeys + 16 + sizeof(float) * ((size_t)alpha * group + kTcCols);
}

bool prefill_tc_supported(int head_dim, int group, int alpha) {
  return head_dim == 128 && group >= 1 && group <= 8 && (group & (group - 1)) == 0 &&
         (long long)alpha * group <= kTcMaxColumns;
}

size_t prefill_lse_tc_smem_bytes(int max_blocks) {
  return 1024 + 2 * kTcHalf + kLtKSlots * 2 * kTcHalf + sizeof(uint64_t) * (1 + 2 * kLtKSlots + 4) + 16 +
         sizeof(float2) * 128 + sizeof(int32_t) * (size_t)max_blocks;
}

size_t prefill_lse_smem_bytes(int head_dim, int max_blocks) {
  const size_t tb = 16 * (size_t)head_dim * 2;
  return 1024 + kKSlots * tb + sizeof(uint64_t) * 2 * kKSlots + sizeof(uint32_t) * kKSlots +
         sizeof(int32_t) * (size_t)max_blocks;
}

cudaError_t prefill_device_setup() {
  const int score_max = (int)prefill_score_smem_bytes(128, kPrefillMaxColumns, 1);
  const void* score[] = {(const void*)prefill_score_kernel<128>, (const void*)prefill_score_kernel<64>};
  for (const void* f : score) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, score_max);
    if (e != cudaSuccess) return e;
  }
  {
    const cudaError_t e = cudaFuncSetAttribute((const void*)prefill_score_tc_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)prefill_score_tc_smem_bytes(kTcMaxColumns, 1));
    if (e != cudaSuccess) return e;
  }
  {
    const cudaError_t e = cudaFuncSetAttribute((const void*)prefill_lse_tc_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)prefill_lse_tc_smem_bytes(kPrefillMaxBlocks));
    if (e != cudaSuccess) return e;
  }
  const void* lse[] = {(const void*)prefill_lse_kernel<128>, (const void*)prefill_lse_kernel<64>};
  for (const void* f : lse) {
    const cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)prefill_lse_smem_bytes(128, kPrefillMaxBlocks));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, bool lse_given, cudaStream_t stream) {
  PrefillArgs args = a;
  void* params[] = {&args};
  if (!lse_given && PKV_PREFILL_TCGEN05 && prefill_tc_supported(head_dim, a.G, a.alpha)) {
    const dim3 grid((unsigned)((a.alpha * a.G + 127) / 128), (unsigned)a.Hkv, (unsigned)a.B);
    const cudaError_t e = launch_pdl((const void*)prefill_lse_tc_kernel, grid, dim3(kLtThreads),
                                     prefill_lse_tc_smem_bytes(a.MB), stream, params);
    if (e != cudaSuccess) return e;
  } else if (!lse_given) {
    const dim3 grid((unsigned)((a.alpha * a.G + kLseCols - 1) / kLseCols), (unsigned)a.Hkv, (unsigned)a.B);
    const void* f = head_dim == 128 ? (const void*)prefill_lse_kernel<128> : (const void*)prefill_lse_kernel<64>;
    const cudaError_t e =
        launch_pdl(f, grid, dim3(kLseWarps * 32), prefill_lse_smem_bytes(head_dim, a.MB), stream, params);
    if (e != cudaSuccess) return e;
  }
  if (PKV_PREFILL_TCGEN05 && prefill_tc_supported(head_dim, a.G, a.alpha)) {
    const dim3 grid((unsigned)((a.MB * 16 + kTcKeys - 1) / kTcKeys), (unsigned)a.Hkv, (unsigned)a.B);
    return launch_pdl((const void*)prefill_score_tc_kernel, grid, dim3(kTcThreads),
                      prefill_score_tc_smem_bytes(a.alpha, a.G), stream, params);
  }
  const dim3 grid((unsigned)((a.MB * 16 + kScoreKeys - 1) / kScoreKeys), (unsigned)a.Hkv, (unsigned)a.B);
  const void* f = head_dim == 128 ? (const void*)prefill_score_kernel<128> : (const void*)prefill_score_kernel<64>;
  return launch_pdl(f, grid, dim3(kScoreWarps * 32), prefill_score_smem_bytes(head_dim, a.alpha, a.G), stream,
                    params);
}

}  // namespace pkv
