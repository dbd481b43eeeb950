// kvops.cu -- KV append, kept-token compaction and top-k kept-token selection for sm_103a.
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

// Compaction: compact position j of (b, g) <- source token kept[b][g][j] (the per-layer
// block-table policy of "How KV Sparsity Achieves 1.5x Acceleration for vLLM", section "Key
// technique 1").  One warp per (b, g, j).
template <int D>
__global__ void __launch_bounds__(256) kv_compact_kernel(
    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, const int32_t* __restrict__ dbt,
    int dNB, int dMB, const __nv_bfloat16* __restrict__ sk, const __nv_bfloat16* __restrict__ sv,
    const int32_t* __restrict__ sbt, const int32_t* __restrict__ lens,
    const int32_t* __restrict__ kept, const int32_t* __restrict__ kept_lens, int max_kept, int B,
    int Hkv, int sNB, int sMB, int32_t* err) {
  const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_launch_dependents();
  if (item >= (int64_t)B * Hkv * max_kept) return;
  const int j = (int)(item % max_kept);
  const int64_t bg = item / max_kept;
  const int b = (int)(bg / Hkv);
  const int g = (int)(bg - (int64_t)b * Hkv);
  const int n = __ldg(kept_lens + b);
  if (j >= n) return;
  if (n > max_kept || n > dMB * 16) {
    if (lane == 0) record_error(err, PKV_DEV_BAD_KEPT_INDEX);
    return;
  }
  const int t = __ldg(kept + bg * max_kept + j);
  const int L = __ldg(lens + b);
  if (t < 0 || t >= L || (t >> 4) >= sMB) {
    if (lane == 0) record_error(err, PKV_DEV_BAD_KEPT_INDEX);
    return;
  }
  const int src_blk = __ldg(sbt + (size_t)b * sMB + (t >> 4));
  const int dst_blk = __ldg(dbt + (size_t)b * dMB + (j >> 4));
  if (src_blk < 0 || src_blk >= sNB || dst_blk < 0 || dst_blk >= dNB) {
    if (lane == 0) record_error(err, PKV_DEV_BAD_BLOCK_ID);
    return;
  }
  const size_t src = (((size_t)src_blk * Hkv + g) * 16 + (t & 15)) * D;
  const size_t dst = (((size_t)dst_blk * Hkv + g) * 16 + (j & 15)) * D;
  if (lane < 16) copy_row_half<D>(dk + dst, sk + src, lane);
  else copy_row_half<D>(dv + dst, sv + src, lane - 16);
}

// ---------------------------------------------------------------------------- top-k select

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

// Order-preserving map of an fp32 score to uint32: a larger key is a larger score.  -0.0
// is folded onto +0.0 first so the two compare equal, as the selection rule requires.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one flag per thread; returns the exclusive prefix and sets
// *total.  Uses `warp_sums` (kSelWarps ints) in shared memory.
__device__ __forceinline__ int block_exclusive_scan(int flag, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const unsigned ballot = __ballot_sync(kFullMask, flag);
  const int in_warp = __popc(ballot & ((1u << lane) - 1u));
  if (lane == 0) warp_sums[warp] = __popc(ballot);
  __syncthreads();
  int before = 0, sum = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const int c = warp_sums[w];
    before += (w < warp) ? c : 0;
    sum += c;
  }
  __syncthreads();
  *total = sum;
  return before + in_warp;
}

// Kept-token selection for one (sequence, kv head) per CTA ("How KV Sparsity...": sections
// "System model" -- drop low-score KV, retain high-score and recent KV -- and "2. Attention
// modification" -- per layer and head, the top-k tokens by accumulated score; sink tokens
// from its introduction).  The k_top-th largest key among the candidates is found by an
// MSD radix select (4 passes of 8 bits over a 256-bin histogram); candidates above it are
// kept, and of those equal to it the lowest positions fill the remainder.  The kept list
// is emitted in ascending position order by block-wide scans, so the result is exact.
__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(
    int32_t* __restrict__ kept_out, int32_t* __restrict__ kept_lens_out,
    const float* __restrict__ scores, int stride, const int32_t* __restrict__ lens, int Hkv,
    int n_sink, int n_recent, int k_top, int32_t* err) {
  __shared__ int hist[256];
  __shared__ int warp_sums[kSelWarps];
  __shared__ int s_digit, s_need;

  grid_dependency_wait();
  grid_launch_dependents();
  const int pair = blockIdx.x;
  const int b = pair / Hkv;
  const int g = pair - b * Hkv;
  const int keep_max = n_sink + k_top + n_recent;
  int L = __ldg(lens + b);
  if (L < 0 || L > stride) {
    if (threadIdx.x == 0) record_error(err, PKV_DEV_BAD_CONTEXT_LEN);
    L = 0;
  }
  int32_t* out = kept_out + (size_t)pair * keep_max;
  if (g == 0 && threadIdx.x == 0) kept_lens_out[b] = min(L, keep_max);
  if (L <= keep_max) {
    for (int t = threadIdx.x; t < L; t += blockDim.x) out[t] = t;
    return;
  }
  const float* row = scores + (size_t)pair * stride;
  const int first = n_sink;
  const int last = L - n_recent;  // candidates [first, last)

  uint32_t prefix = 0u;
  int need = k_top;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xffffffffu << (shift + 8));
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int c = first + threadIdx.x; c < last; c += blockDim.x) {
      const float s = __ldg(row + c);
      if (pass == 0 && s != s) record_error(err, PKV_DEV_BAD_SCORE);
      const uint32_t key = (s != s) ? 0u : score_key(s);
      if ((key & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(key >> shift) & 0xffu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // The digit d holding the need-th largest key: count(> d) < need <= count(>= d).
      int cum = 0;
      int digit = 0;
      for (int d = 255; d >= 0; --d) {
        const int c = hist[d];
        if (cum + c >= need) {
          digit = d;
          break;
        }
        cum += c;
      }
      s_digit = digit;
      s_need = need - cum;
    }
    __syncthreads();
    prefix |= (uint32_t)s_digit << shift;
    need = s_need;
    __syncthreads();
  }
  // prefix is the key of the k_top-th best candidate; `need` of the candidates equal to it
  // are kept, the lowest positions first.
  const uint32_t thr = prefix;
  for (int t = threadIdx.x; t < n_sink; t += blockDim.x) out[t] = t;
  int eq_base = 0, sel_base = 0;
  for (int base = first; base < last; base += blockDim.x) {
    const int c = base + threadIdx.x;
    uint32_t key = 0u;
    if (c < last) {
      const float s = __ldg(row + c);
      key = (s != s) ? 0u : score_key(s);
    }
    const bool in = c < last;
    const int eq = in && key == thr;
    int eq_total;
    const int eq_rank = eq_base + block_exclusive_scan(eq, warp_sums, &eq_total);
    eq_base += eq_total;
    const int sel = in && (key > thr || (eq && eq_rank < need));
    int sel_total;
    const int pos = sel_base + block_exclusive_scan(sel, warp_sums, &sel_total);
    sel_base += sel_total;
    if (sel) out[n_sink + pos] = c;
  }
  for (int t = threadIdx.x; t < n_recent; t += blockDim.x) out[n_sink + k_top + t] = last + t;
}

}  // namespace

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

cudaError_t launch_kv_compact(void* dk, void* dv, const int32_t* dbt, int dNB, int dMB,
                              const void* sk, const void* sv, const int32_t* sbt,
                              const int32_t* lens, const int32_t* kept, const int32_t* kept_lens,
                              int max_kept, int B, int Hkv, int D, int sNB, int sMB,
                              int32_t* err, cudaStream_t stream) {
  const int64_t warps = (int64_t)B * Hkv * max_kept;
  if (warps == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  auto* a = static_cast<__nv_bfloat16*>(dk);
  auto* c = static_cast<__nv_bfloat16*>(dv);
  auto* s1 = static_cast<const __nv_bfloat16*>(sk);
  auto* s2 = static_cast<const __nv_bfloat16*>(sv);
  void* args[] = {&a, &c, &dbt, &dNB, &dMB, &s1, &s2, &sbt, &lens, &kept, &kept_lens,
                  &max_kept, &B, &Hkv, &sNB, &sMB, &err};
  const void* fn = D == 128 ? (const void*)kv_compact_kernel<128> : (const void*)kv_compact_kernel<64>;
  return launch_pdl(fn, dim3(grid), dim3(256), 0, stream, args);
}

cudaError_t launch_select_topk(int32_t* kept_out, int32_t* kept_lens_out, const float* scores,
                               int stride, const int32_t* lens, int B, int Hkv, int n_sink,
                               int n_recent, int k_top, int32_t* err, cudaStream_t stream) {
  const int pairs = B * Hkv;
  if (pairs == 0) return cudaSuccess;
  void* args[] = {&kept_out, &kept_lens_out, &scores, &stride, &lens, &Hkv, &n_sink, &n_recent,
                  &k_top, &err};
  return launch_pdl((const void*)select_topk_kernel, dim3(pairs), dim3(kSelThreads), 0, stream, args);
}

}  // namespace pkv
