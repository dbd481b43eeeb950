// kvops.cu -- KV append, kept-token compaction and top-k kept-token selection for sm_103a.
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "pkv.h"

namespace pkv {
namespace {

// Copies one head row (D bf16) with a half-warp: lane r of the half moves D*2/16 bytes.
template <int D>
__device__ __forceinline__ void copy_row_half(__nv_bfloat16* dst, const __nv_bfloat16* src, int r) {
  if constexpr (D == 128) {
    reinterpret_cast<uint4*>(dst)[r] = __ldg(reinterpret_cast<const uint4*>(src) + r);
  } else {
    reinterpret_cast<uint2*>(dst)[r] = __ldg(reinterpret_cast<const uint2*>(src) + r);
  }
}

// KV append ("KV Cache primer", cf-1.com/news/5988169, section 2.2: the decode step only adds
// the new token's K and V): one warp per (token, kv head); lanes 0-15 move the K row, lanes
// 16-31 the V row, 16-byte (d=128) or 8-byte (d=64) accesses.
template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(__nv_bfloat16* __restrict__ kc,
                                                        __nv_bfloat16* __restrict__ vc,
                                                        const __nv_bfloat16* __restrict__ k,
                                                        const __nv_bfloat16* __restrict__ v,
                                                        const int64_t* __restrict__ slots,
                                                        int64_t T, int Hkv, int NB,
                                                        int32_t* err) {
  const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();  // programmatic launch: the previous kernel may still read the pool
  grid_launch_dependents();
  if (item >= T * Hkv) return;
  const int64_t tok = item / Hkv;
  const int g = (int)(item - tok * Hkv);
  const int64_t slot = __ldg(slots + tok);
  if (slot < 0) return;
  if (slot >= (int64_t)NB * 16) {
    if (lane == 0) record_error(err, PKV_DEV_BAD_SLOT);
    return;
  }
  const int64_t blk = slot >> 4;
  const int off = (int)(slot & 15);
  const size_t dst = (((size_t)blk * Hkv + g) * 16 + off) * D;
  const size_t src = ((size_t)tok * Hkv + g) * D;
  if (lane < 16) copy_row_half<D>(kc + dst, k + src, lane);
  else copy_row_half<D>(vc + dst, v + src, lane - 16);
}

// INT8 row rule (the KV-cache primer's INT8 cache, section 4.2): each (token, kv head) row of
// d values gets one fp32 scale s = max|x| / 127 and codes round_half_even(x / s), clamped to
// [-127, 127]; a zero row gets s = 0 and codes 0.  The division and rounding are IEEE single
// precision (they decide the codes).  A code c is stored as the byte c + 128 (so the decode's
// int8-to-fp16 conversion needs no sign flip).  A warp quantizes one token's K row (lanes 0-15) and V
// row (lanes 16-31), D/16 elements a lane, and stores codes and scales at the given rows; if
// either row holds a non-finite value it stores nothing and returns false.  Every lane of the
// warp calls it.
template <int D>
__device__ __forceinline__ bool quantize_kv_rows(uint8_t* kq_row, uint8_t* vq_row, float* ks_at, float* vs_at,
                                                 const __nv_bfloat16* k_src, const __nv_bfloat16* v_src,
                                                 int lane) {
  constexpr int E = D / 16;  // elements per lane
  const int h = lane & 15;
  const __nv_bfloat16* src = (lane < 16 ? k_src : v_src) + h * E;
  float x[E];
  if constexpr (E == 8) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(ws[i] << 16);
      x[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
    }
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x[2 * i] = __uint_as_float(ws[i] << 16);
      x[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
    }
  }
  float amax = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    finite &= isfinite(x[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));  // within the half
  if (!__all_sync(kFullMask, finite)) return false;
  const float sc = __fdiv_rn(amax, 127.0f);
  uint32_t packed[E / 4];
#pragma unroll
  for (int i = 0; i < E / 4; ++i) packed[i] = 0u;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    int c = 0;
    if (sc != 0.f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], sc))));
    packed[i / 4] |= (uint32_t)(c + 128) << (8 * (i % 4));
  }
  uint8_t* dst = (lane < 16 ? kq_row : vq_row) + h * E;
  if constexpr (E == 8)
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  else
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  if (h == 0) *(lane < 16 ? ks_at : vs_at) = sc;
  return true;
}

// INT8 append: the new token's K and V rows quantized into INT8 pools by the row rule above.
// One warp per (token, kv head).  A non-finite element skips the token's rows and is reported.
template <int D>
__global__ void __launch_bounds__(256) kv_append_q8_kernel(uint8_t* __restrict__ kq, uint8_t* __restrict__ vq,
                                                           float* __restrict__ ks, float* __restrict__ vs,
                                                           const __nv_bfloat16* __restrict__ k,
                                                           const __nv_bfloat16* __restrict__ v,
                                                           const int64_t* __restrict__ slots, int64_t T,
                                                           int Hkv, int NB, int32_t* err) {
  const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_launch_dependents();
  if (item >= T * Hkv) return;
  const int64_t tok = item / Hkv;
  const int g = (int)(item - tok * Hkv);
  const int64_t slot = __ldg(slots + tok);
  if (slot < 0) return;
  if (slot >= (int64_t)NB * 16) {
    if (lane == 0) record_error(err, PKV_DEV_BAD_SLOT);
    return;
  }
  const size_t row = ((size_t)(slot >> 4) * Hkv + g) * 16 + (size_t)(slot & 15);
  const size_t src = ((size_t)tok * Hkv + g) * D;
  if (!quantize_kv_rows<D>(kq + row * D, vq + row * D, ks + row, vs + row, k + src, v + src, lane) && lane == 0)
    record_error(err, PKV_DEV_BAD_VALUE);
}

// Compaction: compact position j of (b, g) <- source token kept[b][g][j] (the per-layer
// block-table policy of "How KV Sparsity Achieves 1.5x Acceleration for vLLM", section "Key
// technique 1").  Rows are RB bytes: bf16 rows of 2d bytes, or INT8 rows of d bytes whose fp32
// row scales move with them when SCALES.  One warp per (b, g, compact_rows(RB) consecutive
// compact positions inside one destination block): the lanes resolve the group's positions to source
// rows (kept index, then source block id: one chain of dependent loads for the group instead
// of one per row), then every lane loads its 16-byte chunks of the group's K and V rows (and
// the row scales) before any is stored, and the stores fill consecutive rows of the destination
// block.  EARLY (the caller declared every input final before the preceding work): the warp
// reads all of it before waiting for that work, and waits on every path before its first write
// -- the error word included -- so that the call also ends after the work it follows.
// positions per warp (a divisor of 16): 4 for 256-byte rows, 8 for shorter ones (measured)
__host__ __device__ constexpr int compact_rows(int rb) { return rb >= 256 ? 4 : 8; }

// the last step of a compaction warp: wait for the preceding work if it was not waited for at the
// start, then record this lane's error (0: none)
template <bool EARLY>
__device__ __forceinline__ void compact_finish(int32_t* err, int code) {
  if constexpr (EARLY) grid_dependency_wait();
  if (code != 0) record_error(err, code);
}

template <int RB, bool SCALES, bool EARLY>
__global__ void __launch_bounds__(256) kv_compact_kernel(
    unsigned char* __restrict__ dk, unsigned char* __restrict__ dv, float* __restrict__ dks,
    float* __restrict__ dvs, const int32_t* __restrict__ dbt, int dNB, int dMB,
    const unsigned char* __restrict__ sk, const unsigned char* __restrict__ sv, const float* __restrict__ sks,
    const float* __restrict__ svs, const int32_t* __restrict__ sbt, const int32_t* __restrict__ lens,
    const int32_t* __restrict__ kept, const int32_t* __restrict__ kept_lens, int max_kept, int B,
    int Hkv, int sNB, int sMB, int32_t* err) {
  static_assert(RB == 64 || RB == 128 || RB == 256, "rows of 64, 128 or 256 bytes");
  constexpr int NR = compact_rows(RB);
  constexpr int CPR = RB / 16;             // 16-byte chunks per row
  constexpr int PER = (NR * CPR + 31) / 32;  // chunks of each pool per lane
  static_assert(16 % NR == 0 && NR * CPR >= 32, "a group fills the warp's lanes");
  const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if constexpr (!EARLY) grid_dependency_wait();
  grid_launch_dependents();
  const int groups = (max_kept + NR - 1) / NR;
  if (item >= (int64_t)B * Hkv * groups) {
    compact_finish<EARLY>(err, 0);
    return;
  }
  const int jb = (int)(item % groups);
  const int64_t bg = item / groups;
  const int b = (int)(bg / Hkv);
  const int g = (int)(bg - (int64_t)b * Hkv);
  const int n = __ldg(kept_lens + b);
  const int j0 = jb * NR;
  if (j0 >= n) {
    compact_finish<EARLY>(err, 0);
    return;
  }
  if (n > max_kept || n > dMB * 16) {
    compact_finish<EARLY>(err, lane == 0 ? PKV_DEV_BAD_KEPT_INDEX : 0);
    return;
  }
  const int dst_blk = __ldg(dbt + (size_t)b * dMB + (j0 >> 4));
  const int r = lane % NR;  // this lane's row of the group (lanes r, r + NR, ... share it)
  long long src_row = -1;
  int code = 0;  // this lane's error
  // the kept entry and the one before it: a list must rise strictly (each kept token has one
  // compact slot), so an entry not above its predecessor is reported and not copied
  const bool has = j0 + r < n;
  int t = -1;
  if (has) t = __ldg(kept + bg * max_kept + j0 + r);
  int tp = __shfl_up_sync(kFullMask, t, 1);  // entry j0 + r - 1 for r > 0
  if (r == 0 && has && j0 > 0) tp = __ldg(kept + bg * max_kept + j0 - 1);
  if (has) {
    const int L = __ldg(lens + b);
    if (t < 0 || t >= L || (t >> 4) >= sMB || (j0 + r > 0 && t <= tp)) {
      if (lane < NR) code = PKV_DEV_BAD_KEPT_INDEX;
    } else {
      const int sb = __ldg(sbt + (size_t)b * sMB + (t >> 4));
      if (sb < 0 || sb >= sNB) {
        if (lane < NR) code = PKV_DEV_BAD_BLOCK_ID;
      } else {
        src_row = ((long long)sb * Hkv + g) * 16 + (t & 15);
      }
    }
  }
  if (dst_blk < 0 || dst_blk >= dNB) {
    compact_finish<EARLY>(err, code);
    if (lane == 0) record_error(err, PKV_DEV_BAD_BLOCK_ID);
    return;
  }
  const size_t dst0 = ((size_t)dst_blk * Hkv + g) * 16 + (j0 & 15);  // row of compact position j0
  uint4 kbuf[PER], vbuf[PER];
  uint32_t live = 0u;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int c = i * 32 + lane;
    const long long sr = __shfl_sync(kFullMask, src_row, (c / CPR) % NR);
    if (c < NR * CPR && sr >= 0) {
      live |= 1u << i;
      kbuf[i] = __ldg(reinterpret_cast<const uint4*>(sk + sr * RB) + c % CPR);
      vbuf[i] = __ldg(reinterpret_cast<const uint4*>(sv + sr * RB) + c % CPR);
    }
  }
  float scl = 0.f;  // lanes 0..NR-1: the K row scale of row r; NR..2NR-1: the V row scale
  if constexpr (SCALES) {
    if (lane < 2 * NR && src_row >= 0) scl = lane < NR ? __ldg(sks + src_row) : __ldg(svs + src_row);
  }
  compact_finish<EARLY>(err, code);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int c = i * 32 + lane;
    if ((live >> i) & 1u) {
      reinterpret_cast<uint4*>(dk + (dst0 + c / CPR) * RB)[c % CPR] = kbuf[i];
      reinterpret_cast<uint4*>(dv + (dst0 + c / CPR) * RB)[c % CPR] = vbuf[i];
    }
  }
  if constexpr (SCALES) {
    if (lane < 2 * NR && src_row >= 0) {
      if (lane < NR) dks[dst0 + r] = scl;
      else dvs[dst0 + r] = scl;
    }
  }
}

// ---------------------------------------------------------------------------- top-k select

#ifndef PKV_SEL_THREADS
#define PKV_SEL_THREADS 512  // one sparse layer: 7.98 us against 8.19 us at 1024 threads (256 were slower)
#endif
constexpr int kSelThreads = PKV_SEL_THREADS;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeys = 40960;  // candidates cached in shared memory (160 KiB)
constexpr int kSelBins = 4096;       // 12-bit digits (the last digit has 8 bits)
constexpr int kSelFilt = 4096;       // keys sharing the first digit kept in a short list
constexpr int kSelRank = kSelThreads;  // keys sharing a prefix ranked exactly, one per thread
constexpr int kSelFast = kSelRank;     // threshold bins up to this size take the one-pass path
constexpr int kSelRankLanes = 4;       // one-pass path: threads ranking one key of the bin
constexpr int kSelBatch = 16;        // score loads in flight per thread
// dynamic shared memory: the cached keys
constexpr int kSelDynSmem = kSelSmemKeys * (int)sizeof(uint32_t);

// Order-preserving map of an fp32 score to uint32: a larger key is a larger score.  -0.0
// is folded onto +0.0 first so the two compare equal, as the selection rule requires; NaN
// (invalid input, reported) maps to the smallest key.
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of two ints per thread at once (one set of barriers); returns
// the prefixes in *pa, *pb.  `sums` holds 2 * (kSelWarps + 1) ints of shared memory.
__device__ __forceinline__ void block_exclusive_scan2(int a, int b, int* sums, int* pa, int* pb) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ta = __shfl_up_sync(kFullMask, ia, o);
    const int tb = __shfl_up_sync(kFullMask, ib, o);
    if (lane >= o) {
      ia += ta;
      ib += tb;
    }
  }
  if (lane == 31) {
    sums[2 * warp] = ia;
    sums[2 * warp + 1] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const int wa = lane < kSelWarps ? sums[2 * lane] : 0;
    const int wb = lane < kSelWarps ? sums[2 * lane + 1] : 0;
    int xa = wa, xb = wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ta = __shfl_up_sync(kFullMask, xa, o);
      const int tb = __shfl_up_sync(kFullMask, xb, o);
      if (lane >= o) {
        xa += ta;
        xb += tb;
      }
    }
    __syncwarp();
    if (lane < kSelWarps) {
      sums[2 * lane] = xa - wa;
      sums[2 * lane + 1] = xb - wb;
    }
  }
  __syncthreads();
  *pa = sums[2 * warp] + ia - a;
  *pb = sums[2 * warp + 1] + ib - b;
  __syncthreads();
}

// Block-wide exclusive prefix of one int per thread with a single barrier: warps scan in
// registers, publish their totals in `wsum` (kSelWarps ints), and every warp adds the totals of
// the warps before it.  `wsum` must not be written again before the block's next barrier.
__device__ __forceinline__ int block_exclusive_scan1(int a, int* wsum) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int incl = a;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = lane < warp ? wsum[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(kFullMask, before, o);
  return before + incl - a;
}

// Kept-token selection for one (sequence, kv head) per CTA ("How KV Sparsity...": sections
// "System model" -- drop low-score KV, retain high-score and recent KV -- and "2. Attention
// modification" -- per layer and head, the top-k tokens by accumulated score; sink tokens
// from its introduction).  The k_top-th largest key among the candidates is found by an MSD
// radix select over digits of 12, 12 and 8 bits: the first pass counts every candidate into a
// 4096-bin histogram while the scores load (scores of one layer share few exponents, so bins
// of 12 bits spread the shared-memory atomics that 8-bit bins would pile onto a few addresses).
// Once at most kSelRank candidates share the digits chosen so far, they are gathered and every
// thread ranks one of them against all the others (the k_top-th key x has count(> x) < need <=
// count(>= x)), which replaces the remaining passes; a larger group goes through the next digit
// (over a short list of the first digit's keys when it fits).  Candidates above the k_top-th
// key are kept, and of those equal to it the lowest positions fill the remainder: each thread
// owns a run of consecutive candidates, marks its kept ones in 64-bit masks, and one block scan
// places them, so the kept list is written in ascending position and the result is exact and
// unique.
// Launched with programmatic stream serialisation.  With EARLY (PKV_SELECT_INPUTS_READY) the
// scores and lengths are final before the previous kernel on the stream ends: the CTA loads,
// counts and selects from its scores first and waits for that kernel only before its first
// global write, the kept list (errors found earlier are held until then).  The keys are cached in `cache_keys` words of dynamic
// shared memory (sized to the score rows, so two CTAs can share an SM when the rows are short).
template <bool EARLY>
__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(
    int32_t* __restrict__ kept_out, int32_t* __restrict__ kept_lens_out,
    const float* __restrict__ scores, int stride, const int32_t* __restrict__ lens, int Hkv,
    int n_sink, int n_recent, int k_top, int32_t* err, int cache_keys) {
  extern __shared__ __align__(16) uint32_t s_keys[];  // cache_keys keys when the candidates fit
  __shared__ __align__(16) int hist[kSelBins];
  __shared__ __align__(16) uint32_t s_filt[kSelFilt];        // keys sharing the first digit (when they fit)
  __shared__ uint32_t s_rank[kSelRank];        // keys sharing the prefix, ranked exactly
  __shared__ int warp_sums[2 * (kSelWarps + 1)];
  __shared__ int warp_tot[kSelWarps];          // block_exclusive_scan1's warp totals
  __shared__ uint32_t kept_bits[kSelSmemKeys / 32];  // one-pass path: kept keys of the threshold bin
  __shared__ int s_digit, s_need, s_bin, s_fcount, s_rcount;
  __shared__ uint32_t s_thr;

  // With EARLY the next kernel may launch at once (two selections' CTAs share an SM when the
  // score rows are short); its own wait orders its writes after this one's.
  bool waited = !EARLY;
  if (waited) grid_dependency_wait();
  grid_launch_dependents();
  const int pair = blockIdx.x;
  const int b = pair / Hkv;
  const int g = pair - b * Hkv;
  const int keep_max = n_sink + k_top + n_recent;
  int L = __ldg(lens + b);
  const bool bad_len = L < 0 || L > stride;
  if (bad_len) L = 0;
  int32_t* out = kept_out + (size_t)pair * keep_max;
  const int first = n_sink;
  const int n = L - n_recent - n_sink;  // candidates: positions first .. first + n - 1
  // Before the first global write: the wait (EARLY), then the writes of every path: the error
  // held, the kept count, and the sinks and the recent window (their stores drain while the
  // selection runs).
  auto start_writes = [&]() {
    if (!waited) {
      grid_dependency_wait();
      waited = true;
    }
    if (bad_len && threadIdx.x == 0) record_error(err, PKV_DEV_BAD_CONTEXT_LEN);
    if (g == 0 && threadIdx.x == 0) kept_lens_out[b] = min(L, keep_max);
    if (L <= keep_max) {
      for (int t = threadIdx.x; t < L; t += blockDim.x) out[t] = t;
      return;
    }
    for (int t = threadIdx.x; t < n_sink; t += blockDim.x) out[t] = t;
    for (int t = threadIdx.x; t < n_recent; t += blockDim.x) out[n_sink + k_top + t] = first + n + t;
  };
  if (waited || L <= keep_max || k_top == 0) start_writes();
  if (L <= keep_max || k_top == 0) return;  // every token, or no candidate, is kept
  const float* row = scores + (size_t)pair * stride;
  const bool cached = n <= cache_keys;
  const int lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < kSelBins; i += blockDim.x) hist[i] = 0;
  for (int i = threadIdx.x; i < kSelSmemKeys / 32; i += blockDim.x) kept_bits[i] = 0u;
  if (threadIdx.x == 0) {
    s_fcount = 0;
    s_rcount = 0;
  }
  __syncthreads();
  // The digit holding the need-th largest key among those matching the prefix so far:
  // count(> d) < need <= count(>= d).  Thread t owns the bins [PB r, PB r + PB), r = threads - 1 - t,
  // so an exclusive scan over the threads counts the keys in higher bins.
  uint32_t prefix = 0u;
  int need = k_top;
  auto pick_digit = [&](int shift, int bins) {
    constexpr int PB = kSelBins / kSelThreads;  // bins per thread
    const int r = kSelThreads - 1 - (int)threadIdx.x;
    int c[PB];
#pragma unroll
    for (int j = 0; j < PB; j += 4) {
      int4 h = make_int4(0, 0, 0, 0);
      if (PB * r + j < bins) h = reinterpret_cast<const int4*>(hist)[(PB * r + j) / 4];
      c[j] = h.x; c[j + 1] = h.y; c[j + 2] = h.z; c[j + 3] = h.w;
    }
    int own = 0;
#pragma unroll
    for (int j = 0; j < PB; ++j) own += c[j];
    const int above = block_exclusive_scan1(own, warp_tot);
    if (own > 0 && above < need && need <= above + own) {
      int cum = above;
#pragma unroll
      for (int j = PB - 1; j >= 0; --j) {
        if (cum + c[j] >= need) {
          s_digit = PB * r + j;
          s_need = need - cum;
          s_bin = c[j];
          break;
        }
        cum += c[j];
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s_digit << shift;
    need = s_need;
  };
  bool nan_seen = false;
  const float* cand = row + first;
  // Scores -> order-preserving keys in shared memory, kSelBatch independent loads in flight
  // per thread, counted by their first 12 bits on the way.
  auto take_key = [&](float v, int i) {
    const uint32_t key = score_key(v);
    nan_seen |= v != v;
    if (cached) s_keys[i] = key;
    atomicAdd(&hist[key >> 20], 1);
  };
  if ((reinterpret_cast<uintptr_t>(cand) & 15u) == 0) {
    // 16-byte loads: thread t takes candidates 4 (t + kSelThreads u) .. + 3, kSelBatch / 4 loads in flight
    constexpr int V = kSelBatch / 4;
    const int n4 = n >> 2;
    for (int base = 0; base < n4; base += kSelThreads * V) {
      float4 v[V];
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int i = base + u * kSelThreads + (int)threadIdx.x;
        v[u] = i < n4 ? __ldg(reinterpret_cast<const float4*>(cand) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int i = base + u * kSelThreads + (int)threadIdx.x;
        if (i < n4) {
          const uint4 k4 = make_uint4(score_key(v[u].x), score_key(v[u].y), score_key(v[u].z), score_key(v[u].w));
          nan_seen |= (v[u].x != v[u].x) | (v[u].y != v[u].y) | (v[u].z != v[u].z) | (v[u].w != v[u].w);
          if (cached) reinterpret_cast<uint4*>(s_keys)[i] = k4;  // one 16-byte store
          atomicAdd(&hist[k4.x >> 20], 1);
          atomicAdd(&hist[k4.y >> 20], 1);
          atomicAdd(&hist[k4.z >> 20], 1);
          atomicAdd(&hist[k4.w >> 20], 1);
        }
      }
    }
    for (int i = 4 * n4 + (int)threadIdx.x; i < n; i += blockDim.x) take_key(__ldg(cand + i), i);
  } else {
    for (int base = 0; base < n; base += kSelThreads * kSelBatch) {
      float v[kSelBatch];
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const int i = base + u * kSelThreads + (int)threadIdx.x;
        v[u] = i < n ? __ldg(cand + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const int i = base + u * kSelThreads + (int)threadIdx.x;
        if (i < n) take_key(v[u], i);
      }
    }
  }
  // the selection itself writes only shared memory: with EARLY the wait comes before the
  // kept list is written (begin_output)
  auto begin_output = [&]() {
    if (!waited) start_writes();
    if (nan_seen) record_error(err, PKV_DEV_BAD_SCORE);
  };
  __syncthreads();
  pick_digit(20, kSelBins);

  // Thread t owns candidates [t*C, t*C + C) (C odd: conflict-free shared-memory reads), at most
  // 64 at a time as bit masks (two 32-bit halves).
  int C = (n + blockDim.x - 1) / blockDim.x;
  C |= 1;
  const int c0 = min(n, (int)threadIdx.x * C);
  const int c1 = min(n, c0 + C);

  // One-pass path (the keys cached, at most kSelFast keys in the k_top-th key's first-digit bin
  // d1): one ordered pass marks each thread's keys above bin d1 and gathers the bin's keys with
  // their positions; each of those is ranked against the others (larger key first, then lower
  // position) by kSelRankLanes threads, and the `need` best are set in a bitmap of kept
  // candidates; a block scan then places every thread's kept positions, in ascending order.  The kept set is the general path's: every key above the
  // k_top-th, then the lowest positions among the keys equal to it.
  if (cached && s_bin <= kSelFast) {
    const uint32_t d1 = prefix >> 20;
    const int need1 = need;
    // the bin's keys as (key, ~position): a larger value ranks first, so equal keys go by
    // lower position and every value is distinct
    unsigned long long* s_rk = reinterpret_cast<unsigned long long*>(s_filt);
    uint32_t above[2] = {0u, 0u}, inbin[2] = {0u, 0u};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i0 = c0 + 32 * h, i1 = min(c1, i0 + 32);
#pragma unroll 8
      for (int i = i0; i < i1; ++i) {
        const uint32_t dg = s_keys[i] >> 20;
        above[h] |= (uint32_t)(dg > d1) << (i - i0);
        inbin[h] |= (uint32_t)(dg == d1) << (i - i0);
      }
    }
    // the bin's keys, one reservation per warp
    const int nin = __popc(inbin[0]) + __popc(inbin[1]);
    int incl = nin;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    int at = 0;
    if (lane == 31 && incl > 0) at = atomicAdd(&s_rcount, incl);
    at = __shfl_sync(kFullMask, at, 31) + incl - nin;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t bits = inbin[h];
      while (bits != 0u) {
        const int i = c0 + 32 * h + __ffs(bits) - 1;
        bits &= bits - 1u;
        s_rk[at] = ((unsigned long long)s_keys[i] << 32) | (uint32_t)~i;
        ++at;
      }
    }
    __syncthreads();
    const int m = s_rcount;  // == s_bin
    constexpr int kGroups = kSelThreads / kSelRankLanes;
    const int sub = (int)threadIdx.x & (kSelRankLanes - 1);
    for (int j0 = 0; j0 < m; j0 += kGroups) {  // uniform trip count: the shuffles see every lane
      const int j = j0 + (int)threadIdx.x / kSelRankLanes;
      int r = 0;
      unsigned long long x = 0ull;
      if (j < m) {
        x = s_rk[j];
        int k = sub;
        for (; k + 3 * kSelRankLanes < m; k += 4 * kSelRankLanes) {
          const unsigned long long y0 = s_rk[k], y1 = s_rk[k + kSelRankLanes];
          const unsigned long long y2 = s_rk[k + 2 * kSelRankLanes], y3 = s_rk[k + 3 * kSelRankLanes];
          r += (int)(y0 > x) + (int)(y1 > x) + (int)(y2 > x) + (int)(y3 > x);
        }
        for (; k < m; k += kSelRankLanes) r += (int)(s_rk[k] > x);
      }
#pragma unroll
      for (int o = 1; o < kSelRankLanes; o <<= 1) r += __shfl_xor_sync(kFullMask, r, o);
      if (j < m && sub == 0 && r < need1) {
        const int px = (int)~(uint32_t)x;
        atomicOr(&kept_bits[px >> 5], 1u << (px & 31));
      }
    }
    __syncthreads();
    // the bitmap's bits of [start, start + 32), start >= 0 (bits past n are zero or unread)
    auto bits32 = [&](int start) -> uint32_t {
      const int w = start >> 5, sh = start & 31;
      const uint32_t lo = kept_bits[w] >> sh;
      return sh == 0 ? lo : lo | (kept_bits[w + 1] << (32 - sh));
    };
    uint32_t take[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) take[h] = above[h] | (inbin[h] != 0u ? inbin[h] & bits32(c0 + 32 * h) : 0u);
    const int cnt = __popc(take[0]) + __popc(take[1]);
    begin_output();
    int w = n_sink + block_exclusive_scan1(cnt, warp_tot);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t t = take[h];
      while (t != 0u) {
        out[w++] = first + c0 + 32 * h + (__ffs(t) - 1);
        t &= t - 1u;
      }
    }
    return;
  }
  auto key_at = [&](int i) -> uint32_t { return cached ? s_keys[i] : score_key(__ldg(row + first + i)); };

  // Gathers the keys of `src` (count m) that share the prefix's top `bits` bits into dst: each
  // warp counts its hits, takes its share of dst with one atomic, then writes them (one
  // reservation per warp: an atomic per hit would serialise the warps on the counter).
  auto gather = [&](const uint32_t* src, int m, int bits, uint32_t* dst, int* count) {
    const uint32_t hi = 0xffffffffu << (32 - bits);
    const uint32_t want = prefix & hi;
    int cnt = 0;
#pragma unroll 4
    for (int base = 0; base < m; base += kSelThreads) {
      const int i = base + (int)threadIdx.x;
      cnt += __popc(__ballot_sync(kFullMask, i < m && (src[i] & hi) == want));
    }
    int at = 0;
    if (lane == 0 && cnt > 0) at = atomicAdd(count, cnt);
    at = __shfl_sync(kFullMask, at, 0);
    if (cnt > 0) {
#pragma unroll 4
      for (int base = 0; base < m; base += kSelThreads) {
        const int i = base + (int)threadIdx.x;
        const uint32_t key = i < m ? src[i] : 0u;
        const bool hit = i < m && (key & hi) == want;
        const unsigned msk = __ballot_sync(kFullMask, hit);
        if (hit) dst[at + __popc(msk & ((1u << lane) - 1u))] = key;
        at += __popc(msk);
      }
    }
    __syncthreads();
  };
  // Counts the next digit (at `shift`, `bins` wide) of the keys sharing the prefix's top
  // `bits` bits, from the short list or from every candidate.
  auto count_digit = [&](const uint32_t* src, int m, int bits, int shift, int bins) {
    for (int i = threadIdx.x; i < kSelBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const uint32_t hi = 0xffffffffu << (32 - bits);
    for (int base = 0; base < m; base += blockDim.x) {
      const int i = base + (int)threadIdx.x;
      const uint32_t key = i < m ? (src != nullptr ? src[i] : key_at(i)) : 0u;
      const bool hit = i < m && (key & hi) == (prefix & hi);
      const int digit = (int)((key >> shift) & (uint32_t)(bins - 1));
      if (src != nullptr) {
        if (hit) atomicAdd(&hist[digit], 1);
      } else {  // every candidate: one atomic per distinct digit of the warp
        const unsigned peers = __match_any_sync(kFullMask, hit ? digit : -1);
        if (hit && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    pick_digit(shift, bins);
  };
  // Exact rank of the (at most kSelRank) keys sharing the prefix's top `bits` bits: the one
  // with count(> x) < need <= count(>= x) is the k_top-th key.
  auto rank_group = [&](const uint32_t* src, int m, int bits) {
    gather(src, m, bits, s_rank, &s_rcount);
    const int mr = s_rcount;
    if ((int)threadIdx.x < mr) {
      const uint32_t x = s_rank[threadIdx.x];
      int gt = 0, ge = 0;
      int j = 0;
      for (; j + 8 <= mr; j += 8) {  // 8 independent (broadcast) loads in flight
        uint32_t y[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = s_rank[j + u];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          gt += y[u] > x;
          ge += y[u] >= x;
        }
      }
      for (; j < mr; ++j) {
        const uint32_t y = s_rank[j];
        gt += y > x;
        ge += y >= x;
      }
      if (gt < need && need <= ge) {  // every thread holding x writes the same values
        s_thr = x;
        s_digit = need - gt;
      }
    }
    __syncthreads();
    prefix = s_thr;
    need = s_digit;
  };

  int bits = 12;
  if (cached && s_bin <= kSelRank) {
    rank_group(s_keys, n, bits);
  } else if (cached && s_bin <= kSelFilt) {
    const int m = s_bin;
    gather(s_keys, n, bits, s_filt, &s_fcount);
    count_digit(s_filt, m, bits, 8, kSelBins);
    bits = 24;
    if (s_bin <= kSelRank) {
      rank_group(s_filt, m, bits);
    } else {
      count_digit(s_filt, m, bits, 0, 256);
    }
  } else {  // too many keys share the first digit for the short list: passes over every key
    count_digit(nullptr, n, bits, 8, kSelBins);
    count_digit(nullptr, n, 24, 0, 256);
  }
  const uint32_t thr = prefix;  // key of the k_top-th best candidate

  // Ordered pass over each thread's candidates, 64 at a time as bit masks (two 32-bit halves)
  // of the keys above thr and equal to it.  A run of at most 64 (always, with the keys cached)
  // keeps its masks for the write.
  auto masks = [&](int i0, uint32_t (&m)[4]) {  // gt lo, gt hi, eq lo, eq hi
    m[0] = m[1] = m[2] = m[3] = 0u;
    const int i1 = min(c1, i0 + 64), mid = min(i1, i0 + 32);
#pragma unroll 8
    for (int i = i0; i < mid; ++i) {
      const uint32_t key = key_at(i);
      m[0] |= (uint32_t)(key > thr) << (i - i0);
      m[2] |= (uint32_t)(key == thr) << (i - i0);
    }
#pragma unroll 8
    for (int i = mid; i < i1; ++i) {
      const uint32_t key = key_at(i);
      m[1] |= (uint32_t)(key > thr) << (i - i0 - 32);
      m[3] |= (uint32_t)(key == thr) << (i - i0 - 32);
    }
  };
  uint32_t mk[4];
  int gt = 0, eq = 0;
  for (int i0 = c0; i0 < c1; i0 += 64) {
    masks(i0, mk);
    gt += __popc(mk[0]) + __popc(mk[1]);
    eq += __popc(mk[2]) + __popc(mk[3]);
  }
  // equal keys are taken lowest position first, so the threads before this one took
  // min(need, eq_before) of them
  int gt_before, eq_before;
  begin_output();
  block_exclusive_scan2(gt, eq, warp_sums, &gt_before, &eq_before);
  int eq_left = max(0, min(eq, need - eq_before));
  int w = n_sink + gt_before + min(need, eq_before);
  if (gt + eq_left > 0) {
    for (int i0 = c0; i0 < c1; i0 += 64) {
      if (c1 - c0 > 64) masks(i0, mk);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t take = mk[h], eqm = mk[2 + h];
        while (eq_left > 0 && eqm != 0u) {  // the lowest remaining equal keys
          take |= eqm & (~eqm + 1u);
          eqm &= eqm - 1u;
          --eq_left;
        }
        while (take != 0u) {
          out[w++] = first + i0 + 32 * h + (__ffs(take) - 1);
          take &= take - 1u;
        }
      }
    }
  }
}

// Rolling admission of a decode step's token into a sparse layer of fixed budget ("How KV
// Sparsity Achieves 1.5x Acceleration for vLLM", section "System model": the layer keeps the
// high-score and the recent KV; the token entering takes the place of the lowest-score one).
// Per (b, kv head g): while the budget is not full the token takes the next slot; when it is,
// the token leaving the recent window (position L - 1 - n_recent) meets the top-k set (slots
// holding positions in [n_sink, that position)): if its score is strictly above the set's
// lowest (ties: the highest position is the weakest), the weakest is dropped, else the leaving
// token is; the new token takes the dropped slot with score 0.  One CTA per sequence, a warp
// per kv head: the warp scans the slots (lane-strided), reduces the leaving slot and the
// weakest (score, position) pair across its lanes, then copies the rows (lanes 0-15 K,
// 16-31 V; with Q8 the rows are quantized into INT8 pools by the row rule of the INT8 append,
// and a non-finite row leaves its (b, g) unchanged).  The slot count is updated after every
// head is done.  EARLY (the caller declared the slot state, lengths and block table final before
// the preceding work): the warps scan and choose their slots before waiting for that work, and
// wait before the step's rows are read and before any write -- the error word included.
constexpr int kAdmitWarps = 8;
constexpr int kAdmitUnroll = 4;  // 16-byte slot loads in flight per lane and per array

template <int D, bool Q8, bool EARLY>
__global__ void __launch_bounds__(kAdmitWarps * 32) kv_rolling_admit_kernel(
    void* __restrict__ kc, void* __restrict__ vc, float* __restrict__ ks, float* __restrict__ vs,
    const int32_t* __restrict__ bt, int NB, int MB, int32_t* __restrict__ slot_pos, float* __restrict__ slot_score,
    int32_t* __restrict__ kept_lens, const int32_t* __restrict__ lens, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, int Hkv, int capacity, int n_sink, int n_recent, int32_t* err) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if constexpr (!EARLY) grid_dependency_wait();
  grid_launch_dependents();
  const int L = lens[b];
  const int used = kept_lens[b];
  const bool valid = L >= 1 && used >= 0 && used <= capacity;
  if constexpr (!EARLY) {
    if (!valid && threadIdx.x == 0) record_error(err, PKV_DEV_BAD_CONTEXT_LEN);
  }
  const bool full = used == capacity;
  for (int g = warp; valid && g < Hkv; g += kAdmitWarps) {
    int32_t* pos = slot_pos + ((size_t)b * Hkv + g) * capacity;
    float* score = slot_score + ((size_t)b * Hkv + g) * capacity;
    int target = used;
    bool ok = true;
    if (full) {
      const int leaving = L - 1 - n_recent;
      int s_out = -1, s_min = -1, p_min = -1;
      float x_min = INFINITY;
      bool nan = false;
      // the weakest top-k token is unique under (score ascending, position descending), so
      // the order in which the lanes visit the slots does not matter
      auto visit = [&](int s, int p, float x) {
        nan |= (x != x);
        if (p == leaving) s_out = s;
        if (p >= n_sink && p < leaving && (s_min < 0 || x < x_min || (x == x_min && p > p_min))) {
          s_min = s;
          x_min = x;
          p_min = p;
        }
      };
      if ((capacity & 3) == 0 && ((reinterpret_cast<uintptr_t>(pos) | reinterpret_cast<uintptr_t>(score)) & 15) == 0) {
        // 16-byte loads, kAdmitUnroll of each issued before any is used
        for (int base = lane * 4; base < capacity; base += 32 * 4 * kAdmitUnroll) {
          int4 pv[kAdmitUnroll];
          float4 xv[kAdmitUnroll];
#pragma unroll
          for (int u = 0; u < kAdmitUnroll; ++u) {
            const int s = base + u * 128;
            if (s < capacity) {
              pv[u] = *reinterpret_cast<const int4*>(pos + s);
              xv[u] = *reinterpret_cast<const float4*>(score + s);
            }
          }
#pragma unroll
          for (int u = 0; u < kAdmitUnroll; ++u) {
            const int s = base + u * 128;
            if (s < capacity) {
              visit(s, pv[u].x, xv[u].x);
              visit(s + 1, pv[u].y, xv[u].y);
              visit(s + 2, pv[u].z, xv[u].z);
              visit(s + 3, pv[u].w, xv[u].w);
            }
          }
        }
      } else {
        for (int s = lane; s < capacity; s += 32) visit(s, pos[s], score[s]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s_out = max(s_out, __shfl_xor_sync(kFullMask, s_out, o));
        const int s2 = __shfl_xor_sync(kFullMask, s_min, o);
        const int p2 = __shfl_xor_sync(kFullMask, p_min, o);
        const float x2 = __shfl_xor_sync(kFullMask, x_min, o);
        if (s2 >= 0 && (s_min < 0 || x2 < x_min || (x2 == x_min && p2 > p_min))) {
          s_min = s2;
          x_min = x2;
          p_min = p2;
        }
      }
      nan = __any_sync(kFullMask, nan);
      if (nan || s_out < 0) {
        if constexpr (EARLY) grid_dependency_wait();
        if (lane == 0) record_error(err, nan ? PKV_DEV_BAD_SCORE : PKV_DEV_BAD_KEPT_INDEX);
        ok = false;
      } else {
        target = (s_min >= 0 && score[s_out] > x_min) ? s_min : s_out;
      }
      __syncwarp();  // every lane has read the scores before lane 0 overwrites one
    }
    if (ok) {
      const int blk = target / 16 < MB ? bt[(size_t)b * MB + target / 16] : -1;
      if constexpr (EARLY) grid_dependency_wait();  // the step's rows, and every write, after it
      if (blk < 0 || blk >= NB) {
        if (lane == 0) record_error(err, PKV_DEV_BAD_BLOCK_ID);
      } else {
        const size_t row = ((size_t)blk * Hkv + g) * 16 + (target & 15);
        const size_t src = ((size_t)b * Hkv + g) * D;
        bool written = true;
        if constexpr (Q8) {
          written = quantize_kv_rows<D>(static_cast<uint8_t*>(kc) + row * D, static_cast<uint8_t*>(vc) + row * D,
                                        ks + row, vs + row, k_new + src, v_new + src, lane);
          if (!written && lane == 0) record_error(err, PKV_DEV_BAD_VALUE);
        } else {
          if (lane < 16) copy_row_half<D>(static_cast<__nv_bfloat16*>(kc) + row * D, k_new + src, lane);
          else copy_row_half<D>(static_cast<__nv_bfloat16*>(vc) + row * D, v_new + src, lane - 16);
        }
        if (written && lane == 0) {
          pos[target] = L - 1;
          score[target] = 0.f;
        }
      }
    }
  }
  if constexpr (EARLY) {  // every thread waits, so the call also ends after the work it follows
    grid_dependency_wait();
    if (!valid && threadIdx.x == 0) record_error(err, PKV_DEV_BAD_CONTEXT_LEN);
  }
  __syncthreads();
  if (threadIdx.x == 0 && valid && !full) kept_lens[b] = used + 1;
}

}  // namespace

cudaError_t kvops_device_setup() {
  // the selection's key cache needs more than the default 48 KiB of dynamic shared memory
  cudaError_t e = cudaFuncSetAttribute((const void*)select_topk_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSelDynSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute((const void*)select_topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSelDynSmem);
}

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                             const int64_t* slots, int64_t T, int Hkv, int D, int NB,
                             int32_t* err, cudaStream_t stream) {
  const int64_t warps = T * Hkv;
  if (warps == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  auto* kc = static_cast<__nv_bfloat16*>(k_cache);
  auto* vc = static_cast<__nv_bfloat16*>(v_cache);
  auto* kk = static_cast<const __nv_bfloat16*>(k);
  auto* vv = static_cast<const __nv_bfloat16*>(v);
  void* args[] = {&kc, &vc, &kk, &vv, &slots, &T, &Hkv, &NB, &err};
  const void* fn = D == 128 ? (const void*)kv_append_kernel<128> : (const void*)kv_append_kernel<64>;
  return launch_pdl(fn, dim3(grid), dim3(256), 0, stream, args);
}

cudaError_t launch_kv_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                                const void* k, const void* v, const int64_t* slots, int64_t T, int Hkv,
                                int D, int NB, int32_t* err, cudaStream_t stream) {
  const int64_t warps = T * Hkv;
  if (warps == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  auto* kq = static_cast<uint8_t*>(k_codes);
  auto* vq = static_cast<uint8_t*>(v_codes);
  auto* kk = static_cast<const __nv_bfloat16*>(k);
  auto* vv = static_cast<const __nv_bfloat16*>(v);
  void* args[] = {&kq, &vq, &k_scales, &v_scales, &kk, &vv, &slots, &T, &Hkv, &NB, &err};
  const void* fn = D == 128 ? (const void*)kv_append_q8_kernel<128> : (const void*)kv_append_q8_kernel<64>;
  return launch_pdl(fn, dim3(grid), dim3(256), 0, stream, args);
}

cudaError_t launch_kv_compact(void* dk, void* dv, const int32_t* dbt, int dNB, int dMB,
                              const void* sk, const void* sv, const int32_t* sbt,
                              const int32_t* lens, const int32_t* kept, const int32_t* kept_lens,
                              int max_kept, int B, int Hkv, int D, int sNB, int sMB, int early,
                              int32_t* err, cudaStream_t stream) {
  return launch_kv_compact_q8(dk, dv, nullptr, nullptr, dbt, dNB, dMB, sk, sv, nullptr, nullptr, sbt, lens,
                              kept, kept_lens, max_kept, B, Hkv, D, sNB, sMB, early, err, stream);
}

cudaError_t launch_kv_compact_q8(void* dk, void* dv, float* dks, float* dvs, const int32_t* dbt, int dNB,
                                 int dMB, const void* sk, const void* sv, const float* sks, const float* svs,
                                 const int32_t* sbt, const int32_t* lens, const int32_t* kept,
                                 const int32_t* kept_lens, int max_kept, int B, int Hkv, int D, int sNB,
                                 int sMB, int early, int32_t* err, cudaStream_t stream) {
  const int nr = compact_rows(dks != nullptr ? D : 2 * D);
  const int64_t warps = (int64_t)B * Hkv * ((max_kept + nr - 1) / nr);
  if (warps == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  auto* a = static_cast<unsigned char*>(dk);
  auto* c = static_cast<unsigned char*>(dv);
  auto* s1 = static_cast<const unsigned char*>(sk);
  auto* s2 = static_cast<const unsigned char*>(sv);
  void* args[] = {&a, &c, &dks, &dvs, &dbt, &dNB, &dMB, &s1, &s2, &sks, &svs, &sbt, &lens, &kept, &kept_lens,
                  &max_kept, &B, &Hkv, &sNB, &sMB, &err};
  const bool q8 = dks != nullptr;
  const void* fn;
  if (early)
    fn = q8 ? (D == 128 ? (const void*)kv_compact_kernel<128, true, true> : (const void*)kv_compact_kernel<64, true, true>)
            : (D == 128 ? (const void*)kv_compact_kernel<256, false, true>
                        : (const void*)kv_compact_kernel<128, false, true>);
  else
    fn = q8 ? (D == 128 ? (const void*)kv_compact_kernel<128, true, false>
                        : (const void*)kv_compact_kernel<64, true, false>)
            : (D == 128 ? (const void*)kv_compact_kernel<256, false, false>
                        : (const void*)kv_compact_kernel<128, false, false>);
  return launch_pdl(fn, dim3(grid), dim3(256), 0, stream, args);
}

cudaError_t launch_select_topk(int32_t* kept_out, int32_t* kept_lens_out, const float* scores,
                               int stride, const int32_t* lens, int B, int Hkv, int n_sink,
                               int n_recent, int k_top, int early, int32_t* err, cudaStream_t stream) {
  const int pairs = B * Hkv;
  if (pairs == 0) return cudaSuccess;
  // Flagged calls size the key cache to a score row (the candidates are fewer), up to
  // kSelSmemKeys, so that a call's CTAs can share SMs with the previous call's and select while it
  // finishes; unflagged calls keep one CTA per SM (two of one call on an SM would share its issue
  // slots while other SMs idle: 16 sparse layers 8.96 -> 9.21 us per selection, measured).
  int cache_keys = early ? std::min((stride + 3) & ~3, kSelSmemKeys) : kSelSmemKeys;
  void* args[] = {&kept_out, &kept_lens_out, &scores, &stride, &lens, &Hkv, &n_sink, &n_recent,
                  &k_top, &err, &cache_keys};
  return launch_pdl(early ? (const void*)select_topk_kernel<true> : (const void*)select_topk_kernel<false>,
                    dim3(pairs), dim3(kSelThreads), (size_t)cache_keys * sizeof(uint32_t), stream, args);
}

cudaError_t launch_kv_rolling_admit(void* k_cache, void* v_cache, const int32_t* bt, int NB, int MB,
                                    int32_t* slot_pos, float* slot_score, int32_t* kept_lens,
                                    const int32_t* lens, const void* k_new, const void* v_new, int B,
                                    int Hkv, int D, int capacity, int n_sink, int n_recent, int early,
                                    int32_t* err, cudaStream_t stream) {
  return launch_kv_rolling_admit_q8(k_cache, v_cache, nullptr, nullptr, bt, NB, MB, slot_pos, slot_score,
                                    kept_lens, lens, k_new, v_new, B, Hkv, D, capacity, n_sink, n_recent, early,
                                    err, stream);
}

cudaError_t launch_kv_rolling_admit_q8(void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                       const int32_t* bt, int NB, int MB, int32_t* slot_pos, float* slot_score,
                                       int32_t* kept_lens, const int32_t* lens, const void* k_new,
                                       const void* v_new, int B, int Hkv, int D, int capacity, int n_sink,
                                       int n_recent, int early, int32_t* err, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  auto* kn = static_cast<const __nv_bfloat16*>(k_new);
  auto* vn = static_cast<const __nv_bfloat16*>(v_new);
  void* args[] = {&k_cache, &v_cache, &k_scales, &v_scales, &bt, &NB, &MB, &slot_pos, &slot_score, &kept_lens,
                  &lens, &kn, &vn, &Hkv, &capacity, &n_sink, &n_recent, &err};
  const bool q8 = k_scales != nullptr;
  const void* fn;
  if (early)
    fn = q8 ? (D == 128 ? (const void*)kv_rolling_admit_kernel<128, true, true>
                        : (const void*)kv_rolling_admit_kernel<64, true, true>)
            : (D == 128 ? (const void*)kv_rolling_admit_kernel<128, false, true>
                        : (const void*)kv_rolling_admit_kernel<64, false, true>);
  else
    fn = q8 ? (D == 128 ? (const void*)kv_rolling_admit_kernel<128, true, false>
                        : (const void*)kv_rolling_admit_kernel<64, true, false>)
            : (D == 128 ? (const void*)kv_rolling_admit_kernel<128, false, false>
                        : (const void*)kv_rolling_admit_kernel<64, false, false>);
  return launch_pdl(fn, dim3(B), dim3(kAdmitWarps * 32), 0, stream, args);
}

}  // namespace pkv
