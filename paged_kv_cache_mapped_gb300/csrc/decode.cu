// decode.cu -- single-token decode attention over a paged KV cache, for sm_103a.
//
// out[b,h] = softmax(scale * q[b,h] . K_t) . V_t over the attended tokens t of sequence b
// (the attention formula of "Transformer模型中的KV Cache优化推理策略", yutianautomatic.com,
// evaluated for one new query against the cached K/V as the KV-cache primer,
// cf-1.com/news/5988169, section 2.2 describes; K/V found through the block table of its
// section 4.1).  Dense mode attends [max(0, L-window), L); sparse mode attends a kept list
// (the layer-wise sparse variant of "How KV Sparsity Achieves 1.5x Acceleration for vLLM").
//
// Design (GB300-first; HBM-bound, 4-6 flop per KV byte):
//  * Work partition ("stream-K" split): the (sequence, kv head, 16-token unit) list is
//    flattened and cut into equal contiguous ranges, one per worker warp of a persistent
//    grid sized to the SMs, so every SM streams the same number of bytes whatever the
//    length mix.  A range may end inside a (sequence, head) segment: each worker emits a
//    partial (running max m, running sum l, unnormalised o) per segment it touches; a
//    segment covered by one worker writes its output directly.
//  * Each worker warp owns a ring of K/V tile pairs in shared memory.  One lane issues TMA
//    bulk copies (cp.async.bulk, 4 KiB per tile at d=128, L2 evict-first) completing on a
//    per-slot mbarrier; the warp consumes slots in order and refills a slot once every lane
//    has finished reading it.  Sparse mode gathers rows instead: 32 lanes each issue one
//    row copy (16 K rows + 16 V rows) into the same tile layout.
//  * GQA: the G query heads sharing a kv head are processed together, so each K/V byte is
//    read from HBM once per kv head.
//  * Math in fp32 on CUDA cores with Blackwell packed fp32x2 FMA: lane (half, es) holds 8
//    (d=128) or 4 (d=64) elements of q for the G heads and the same slice of the output.
//    Tokens alternate between the two half-warps.  Partial dot products are finished by a
//    butterfly reduce-scatter over the 16 lanes of a half-warp (each lane ends with whole
//    logits of one head), then the online-softmax update ("How KV Sparsity...", section
//    "2. Attention modification", Fig. 7: running max, running sum, rescale, divide at the
//    end) happens in base 2 with log2(e) folded into q.
//  * Every wait is bounded (globaltimer); a timeout records PKV_DEV_WAIT_TIMEOUT, waits for
//    the copies in flight and returns.  Bad block ids / kept indices are skipped and
//    recorded, never dereferenced.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "pkv.h"

namespace pkv {
namespace {

template <int D>
struct Geo {
  static constexpr int kEPL = D / 16;       // bf16 elements of a row held by one lane
  static constexpr int kPairs = kEPL / 2;   // fp32 pairs per lane per row
  static constexpr int kRow = D * 2;        // bytes per K/V row
  static constexpr int kTile = 16 * kRow;   // bytes per 16-token tile
  static constexpr int kRing = (D == 128) ? 3 : 5;
};

template <int G>
struct Grp {
  static constexpr int kGP = G == 1 ? 1 : (G == 2 ? 2 : (G <= 4 ? 4 : 8));  // padded group
  static constexpr int kN = kGP * 8;                     // partial logits per lane per tile
  static constexpr int kVPL = kN >= 16 ? kN / 16 : 1;    // whole logits per lane after reduction
  static constexpr int kLPG = kN >= 16 ? 8 / kVPL : 16;  // lanes of a half-warp sharing one head
};

template <int D, int G>
struct WarpSmem {
  alignas(128) unsigned char tiles[Geo<D>::kRing][2][Geo<D>::kTile];
  uint64_t p2[2 * 8 * Grp<G>::kGP];  // (p, p) pairs, [half][token index][head]
  uint64_t a2[Grp<G>::kGP];          // (alpha, alpha) per head
  float2 ml[Grp<G>::kGP];            // (m, l) per head, at flush
  uint64_t bar[Geo<D>::kRing];
  uint32_t meta[Geo<D>::kRing];      // valid-token mask of the unit held by a slot
};

struct Cursor {
  int b, g, j;  // sequence, kv head, unit within the (b, g) segment
};

__device__ __forceinline__ Cursor locate(int u, const int32_t* s_start, const int32_t* s_nb, int B) {
  int lo = 0, hi = B;  // largest b with s_start[b] <= u; it has units since u < total
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_start[mid] <= u) lo = mid; else hi = mid;
  }
  Cursor c;
  c.b = lo;
  const int nb = s_nb[lo];
  const int rem = u - s_start[lo];
  c.g = rem / nb;
  c.j = rem - c.g * nb;
  return c;
}

__device__ __forceinline__ void advance(Cursor& c, const int32_t* s_nb, int B, int Hkv) {
  if (++c.j == s_nb[c.b]) {
    c.j = 0;
    if (++c.g == Hkv) {
      c.g = 0;
      do { ++c.b; } while (c.b < B && s_nb[c.b] == 0);
    }
  }
}

template <int EPL>
__device__ __forceinline__ void load_row(const unsigned char* p, uint32_t (&w)[EPL / 2]) {
  if constexpr (EPL == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  }
}

// One level of the butterfly reduce-scatter across lanes differing in bit `M` of `es`:
// of the `n` live values, the lane keeps the upper half when its bit is set (else the
// lower half), adds the partner lane's copy of that half, and ends with n/2 live values.
// With a single live value the level is a plain all-reduce.
template <int n, int M, int CAP>
__device__ __forceinline__ void rs_level(float (&v)[CAP], int es) {
  if constexpr (n >= 2) {
    const bool upper = (es & M) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = upper ? v[j] : v[j + n / 2];
      const float keep = upper ? v[j + n / 2] : v[j];
      v[j] = keep + __shfl_xor_sync(kFullMask, send, M);
    }
  } else {
    v[0] += __shfl_xor_sync(kFullMask, v[0], M);
  }
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  const float2 f = unpack2(v);
  return pack2(__shfl_xor_sync(kFullMask, f.x, m), __shfl_xor_sync(kFullMask, f.y, m));
}

template <int D, int G, bool SPARSE>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_split_kernel(const DecodeArgs a) {
  using GE = Geo<D>;
  using GR = Grp<G>;
  constexpr int R = GE::kRing;
  constexpr int EPL = GE::kEPL;
  constexpr int NP = GE::kPairs;
  constexpr int GP = GR::kGP;
  constexpr int N = GR::kN;
  constexpr int VPL = GR::kVPL;
  constexpr int LPG = GR::kLPG;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto* warps_smem = reinterpret_cast<WarpSmem<D, G>*>(smem_raw);
  int32_t* s_start = reinterpret_cast<int32_t*>(smem_raw + sizeof(WarpSmem<D, G>) * kDecodeWarps);
  int32_t* s_nb = s_start + (a.B + 1);
  int32_t* s_first = s_nb + a.B;
  int32_t* s_lo = s_first + a.B;   // dense: first attended token; sparse: context length
  int32_t* s_len = s_lo + a.B;     // dense: context length; sparse: kept count

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int es = lane & 15;
  WarpSmem<D, G>& W = warps_smem[warp];

  // ---- per-sequence unit counts and partition (identical in every CTA) -------------------
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    int L = a.context_lens[b];
    if (L < 0 || L > a.MB * 16) {
      if (blockIdx.x == 0) record_error(a.err, PKV_DEV_BAD_CONTEXT_LEN);
      L = 0;
    }
    int nb, first, lo, len;
    if constexpr (SPARSE) {
      int n = a.kept_lens[b];
      if (n < 0 || n > a.max_kept) {
        if (blockIdx.x == 0) record_error(a.err, PKV_DEV_BAD_KEPT_INDEX);
        n = 0;
      }
      nb = (n + 15) >> 4;
      first = 0;
      lo = L;
      len = n;
    } else {
      lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
      first = lo >> 4;
      nb = L > 0 ? ((L - 1) >> 4) - first + 1 : 0;
      len = L;
    }
    s_nb[b] = nb;
    s_first[b] = first;
    s_lo[b] = lo;
    s_len[b] = len;
  }
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(&W.bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.B; base += 32) {
      const int b = base + lane;
      const int v = (b < a.B) ? s_nb[b] * a.Hkv : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += t;
      }
      if (b < a.B) s_start[b] = carry + incl - v;
      carry += __shfl_sync(kFullMask, incl, 31);
    }
    if (lane == 0) s_start[a.B] = carry;
  }
  __syncthreads();

  const int total = s_start[a.B];
  const long long nworkers = (long long)gridDim.x * kDecodeWarps;
  int per = (int)((total + nworkers - 1) / nworkers);
  if (per < a.min_units) per = a.min_units;
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= a.B; i += blockDim.x) a.layout[2 + i] = s_start[i];
    for (int i = threadIdx.x; i < a.B; i += blockDim.x) a.layout[3 + a.B + i] = s_nb[i];
    if (threadIdx.x == 0) {
      a.layout[0] = total;
      a.layout[1] = per;
    }
  }
  const long long gw = (long long)blockIdx.x * kDecodeWarps + warp;
  if (gw * per >= total) return;  // no __syncthreads after this point
  const int u0 = (int)(gw * per);
  const int nunits = min(total - u0, per);

  const uint64_t pol = l2_policy_evict_first();

  // ---- producer side (issue a unit into a slot) -----------------------------------------
  Cursor ic = locate(u0, s_start, s_nb, a.B);
  Cursor cc = ic;
  int pend_phys = -1;  // dense: block id of the unit `ic` names, loaded one issue ahead
  if constexpr (!SPARSE) {
    if (lane == 0) pend_phys = __ldg(a.block_tables + (size_t)ic.b * a.MB + s_first[ic.b] + ic.j);
  }

  auto issue = [&](int k) {
    const int slot = k % R;
    fence_proxy_async_smem();
    if constexpr (!SPARSE) {
      if (lane == 0) {
        const int phys = pend_phys;
        if (phys < 0 || phys >= a.NB) {
          record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
          W.meta[slot] = 0u;
          mbar_arrive_expect_tx(&W.bar[slot], 0);
        } else {
          W.meta[slot] = 1u;
          mbar_arrive_expect_tx(&W.bar[slot], 2 * GE::kTile);
          const size_t off = ((size_t)phys * a.Hkv + ic.g) * 16 * D;
          bulk_g2s(W.tiles[slot][0], a.k_cache + off, GE::kTile, &W.bar[slot], pol);
          bulk_g2s(W.tiles[slot][1], a.v_cache + off, GE::kTile, &W.bar[slot], pol);
        }
      }
      advance(ic, s_nb, a.B, a.Hkv);
      if (lane == 0 && k + 1 < nunits)
        pend_phys = __ldg(a.block_tables + (size_t)ic.b * a.MB + s_first[ic.b] + ic.j);
    } else {
      const int r = lane & 15;
      const int pos = ic.j * 16 + r;
      bool ok = pos < s_len[ic.b];
      int t = 0, phys = 0;
      if (ok) {
        t = __ldg(a.kept + ((size_t)ic.b * a.Hkv + ic.g) * a.max_kept + pos);
        if (t < 0 || t >= s_lo[ic.b]) {
          record_error(a.err, PKV_DEV_BAD_KEPT_INDEX);
          ok = false;
        }
      }
      if (ok) {
        phys = __ldg(a.block_tables + (size_t)ic.b * a.MB + (t >> 4));
        if (phys < 0 || phys >= a.NB) {
          record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
          ok = false;
        }
      }
      const uint32_t vmask = __ballot_sync(kFullMask, ok) & 0xffffu;
      if (lane == 0) {
        W.meta[slot] = vmask;
        mbar_arrive_expect_tx(&W.bar[slot], 2u * __popc(vmask) * GE::kRow);
      }
      __syncwarp();
      if (ok) {
        const size_t off = (((size_t)phys * a.Hkv + ic.g) * 16 + (t & 15)) * D;
        const __nv_bfloat16* src = (lane >= 16 ? a.v_cache : a.k_cache) + off;
        bulk_g2s(W.tiles[slot][lane >> 4] + r * GE::kRow, src, GE::kRow, &W.bar[slot], pol);
      }
      advance(ic, s_nb, a.B, a.Hkv);
    }
  };

  int issued = 0;
  for (; issued < nunits && issued < R; ++issued) issue(issued);

  // ---- consumer state --------------------------------------------------------------------
  uint64_t q2[G][NP];
  uint64_t o2[G][NP];
  float m_run = -INFINITY, l_run = 0.f;
  const int my_head = es / LPG;  // head (within the group) whose logits this lane finishes
  int seg_b = -1, seg_g = -1, part = 0, nparts = 0;

  auto flush = [&]() {
    float l = l_run;
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) l += __shfl_xor_sync(kFullMask, l, m);
    l += __shfl_xor_sync(kFullMask, l, 16);
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int k = 0; k < NP; ++k) o2[gg][k] = fadd2(o2[gg][k], shfl_xor64(o2[gg][k], 16));
    if (half == 0 && (es % LPG) == 0 && my_head < G) W.ml[my_head] = make_float2(m_run, l);
    __syncwarp();
    if (half == 0) {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float2 ml = W.ml[gg];
        const size_t row = (size_t)seg_b * a.Hq + (size_t)seg_g * G + gg;
        if (nparts == 1) {
          const float inv = ml.y > 0.f ? 1.f / ml.y : 0.f;
          uint32_t packed[NP];
#pragma unroll
          for (int k = 0; k < NP; ++k) {
            const float2 f = unpack2(o2[gg][k]);
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(f.x * inv, f.y * inv);
            packed[k] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          __nv_bfloat16* dst = a.out + row * D + es * EPL;
          if constexpr (EPL == 8)
            *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          else
            *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
        } else {
          float* dst = a.part_o + (row * a.max_parts + part) * D + es * EPL;
#pragma unroll
          for (int k = 0; k < NP; ++k) reinterpret_cast<float2*>(dst)[k] = unpack2(o2[gg][k]);
          if (es == 0) a.part_ml[row * a.max_parts + part] = ml;
        }
      }
    }
    __syncwarp();
  };

  auto begin_segment = [&](const Cursor& c) {
    seg_b = c.b;
    seg_g = c.g;
    const int nb = s_nb[c.b];
    const int seg_begin = s_start[c.b] + c.g * nb;
    const int w0 = seg_begin / per;
    nparts = (seg_begin + nb - 1) / per - w0 + 1;
    part = (int)gw - w0;
    const uint64_t sc = pack2(a.scale_log2, a.scale_log2);
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const unsigned char* qp = reinterpret_cast<const unsigned char*>(
          a.q + ((size_t)c.b * a.Hq + (size_t)c.g * G + gg) * D + es * EPL);
      uint32_t w[NP];
      load_row<EPL>(qp, w);
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        q2[gg][k] = fmul2(bf16x2_to_f32x2(w[k]), sc);
        o2[gg][k] = 0ull;
      }
    }
    m_run = -INFINITY;
    l_run = 0.f;
  };

  bool aborted = false;
  int k = 0;
  for (; k < nunits; ++k) {
    if (cc.b != seg_b || cc.g != seg_g) {
      if (seg_b >= 0) flush();
      begin_segment(cc);
    }
    const int slot = k % R;
    // every lane waits (acquiring the TMA writes); the give-up decision is warp-uniform
    const bool landed = mbar_wait_bounded(&W.bar[slot], (uint32_t)(k / R) & 1u, a.timeout_ns);
    if (!__all_sync(kFullMask, landed)) {
      if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    uint32_t mask;
    if constexpr (SPARSE) {
      mask = W.meta[slot];
    } else {
      const int tok0 = (s_first[cc.b] + cc.j) * 16;
      const int lo = max(s_lo[cc.b] - tok0, 0);
      const int hi = min(s_len[cc.b] - tok0, 16);
      mask = W.meta[slot] ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
    }
    if (mask != 0u) {
      const unsigned char* kt = W.tiles[slot][0] + es * EPL * 2;
      const unsigned char* vt = W.tiles[slot][1] + es * EPL * 2;
      // -- logits: partial dot products of this lane's slice for its 8 tokens -------------
      float v[N];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = 2 * i + half;
        uint32_t w[NP];
        load_row<EPL>(kt + t * GE::kRow, w);
        uint64_t kf[NP];
#pragma unroll
        for (int kk = 0; kk < NP; ++kk) kf[kk] = bf16x2_to_f32x2(w[kk]);
#pragma unroll
        for (int gg = 0; gg < GP; ++gg) {
          if (gg < G) {
            uint64_t acc = ffma2(q2[gg][0], kf[0], 0ull);
#pragma unroll
            for (int kk = 1; kk < NP; ++kk) acc = ffma2(q2[gg][kk], kf[kk], acc);
            const float2 f = unpack2(acc);
            v[gg * 8 + i] = f.x + f.y;
          } else {
            v[gg * 8 + i] = 0.f;
          }
        }
      }
      // -- butterfly reduce-scatter over the 16 lanes of the half-warp -------------------
      rs_level<N, 8>(v, es);
      rs_level<(N >= 2 ? N / 2 : 1), 4>(v, es);
      rs_level<(N >= 4 ? N / 4 : 1), 2>(v, es);
      rs_level<(N >= 8 ? N / 8 : 1), 1>(v, es);
      // -- mask, block max, online-softmax update ----------------------------------------
      float bmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int f = (N >= 16) ? es * VPL + j : (es >> 1);
        const int t = 2 * (f & 7) + half;
        const bool ok = ((mask >> t) & 1u) && (f >> 3) < G;
        v[j] = ok ? v[j] : -INFINITY;
        bmax = fmaxf(bmax, v[j]);
      }
#pragma unroll
      for (int m = 1; m < LPG; m <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(kFullMask, bmax, m));
      bmax = fmaxf(bmax, __shfl_xor_sync(kFullMask, bmax, 16));
      const float m_new = fmaxf(m_run, bmax);
      const float mref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run - mref);
      const bool dup = (N < 16) && (es & 1);  // G == 1: lanes es, es^1 hold the same logit
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const float p = exp2f(v[j] - mref);
        const int f = (N >= 16) ? es * VPL + j : (es >> 1);
        if (!dup && (f >> 3) < G) {
          W.p2[(half * 8 + (f & 7)) * GP + (f >> 3)] = pack2(p, p);
          psum += p;
        }
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (half == 0 && (es % LPG) == 0 && my_head < G) W.a2[my_head] = pack2(alpha, alpha);
      __syncwarp();
      // -- rescale and accumulate P.V for this lane's 8 tokens -------------------------------
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const uint64_t a2 = W.a2[gg];
#pragma unroll
        for (int kk = 0; kk < NP; ++kk) o2[gg][kk] = fmul2(o2[gg][kk], a2);
      }
      const bool partial = mask != 0xffffu;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = 2 * i + half;
        uint32_t w[NP];
        load_row<EPL>(vt + t * GE::kRow, w);
        if (partial && !((mask >> t) & 1u)) {
#pragma unroll
          for (int kk = 0; kk < NP; ++kk) w[kk] = 0u;
        }
        uint64_t vf[NP];
#pragma unroll
        for (int kk = 0; kk < NP; ++kk) vf[kk] = bf16x2_to_f32x2(w[kk]);
        const uint64_t* prow = W.p2 + (half * 8 + i) * GP;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const uint64_t pp = prow[gg];
#pragma unroll
          for (int kk = 0; kk < NP; ++kk) o2[gg][kk] = ffma2(pp, vf[kk], o2[gg][kk]);
        }
      }
    }
    __syncwarp();
    if (issued < nunits) {
      issue(issued);
      ++issued;
    }
    advance(cc, s_nb, a.B, a.Hkv);
  }

  if (aborted) {
    for (int kk = k; kk < issued; ++kk) (void)mbar_wait_bounded(&W.bar[kk % R], (uint32_t)(kk / R) & 1u, a.timeout_ns);
    return;
  }
  flush();
}

// Log-sum-exp merge of the partials of every (sequence, query head) row that more than one
// worker touched; also writes the zero row of empty sequences.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
decode_merge_kernel(const DecodeArgs a, int group) {
  constexpr int EPW = D / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kMergeWarps + warp;
  if (row >= a.B * a.Hq) return;
  const int b = row / a.Hq;
  const int g = (row % a.Hq) / group;
  const int per = a.layout[1];
  const int nb = a.layout[3 + a.B + b];
  __nv_bfloat16* dst = a.out + (size_t)row * D + lane * EPW;
  if (nb == 0) {
#pragma unroll
    for (int e = 0; e < EPW; ++e) dst[e] = __float2bfloat16_rn(0.f);
    return;
  }
  const int seg = a.layout[2 + b] + g * nb;
  const int w0 = seg / per;
  const int np = (seg + nb - 1) / per - w0 + 1;
  if (np == 1) return;
  const float2* ml = a.part_ml + (size_t)row * a.max_parts;
  const float* po = a.part_o + (size_t)row * a.max_parts * D + lane * EPW;
  float M = -INFINITY;
  for (int p = lane; p < np; p += 32) M = fmaxf(M, ml[p].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
  const float mref = (M == -INFINITY) ? 0.f : M;
  float L = 0.f;
  for (int p = lane; p < np; p += 32) L += ml[p].y * exp2f(ml[p].x - mref);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFullMask, L, o);
  float acc[EPW];
#pragma unroll
  for (int e = 0; e < EPW; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int p = 0; p < np; ++p) {
    const float w = exp2f(ml[p].x - mref);
    const float* src = po + (size_t)p * D;
    if constexpr (EPW == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src);
      acc[0] += w * x.x; acc[1] += w * x.y;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < EPW; e += 2) {
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

template <int D, int G>
constexpr size_t warp_smem_bytes() { return sizeof(WarpSmem<D, G>); }

}  // namespace

#define PKV_DECODE_CASE(D, G)                                                              \
  if (head_dim == D && group == G)                                                         \
    return sparse ? DecodeKernel{(const void*)decode_split_kernel<D, G, true>,             \
                                 (const void*)decode_merge_kernel<D>, D, G, true}          \
                  : DecodeKernel{(const void*)decode_split_kernel<D, G, false>,            \
                                 (const void*)decode_merge_kernel<D>, D, G, false};

DecodeKernel decode_kernel(int head_dim, int group, bool sparse) {
  PKV_DECODE_CASE(128, 1) PKV_DECODE_CASE(128, 2) PKV_DECODE_CASE(128, 4)
  PKV_DECODE_CASE(128, 6) PKV_DECODE_CASE(128, 8)
  PKV_DECODE_CASE(64, 1) PKV_DECODE_CASE(64, 2) PKV_DECODE_CASE(64, 4)
  PKV_DECODE_CASE(64, 6) PKV_DECODE_CASE(64, 8)
  return DecodeKernel{nullptr, nullptr, head_dim, group, sparse};
}

#define PKV_SMEM_CASE(D, G) \
  if (head_dim == D && group == G) per_warp = warp_smem_bytes<D, G>();

size_t decode_smem_bytes(int head_dim, int group, int batch) {
  size_t per_warp = 0;
  PKV_SMEM_CASE(128, 1) PKV_SMEM_CASE(128, 2) PKV_SMEM_CASE(128, 4) PKV_SMEM_CASE(128, 6)
  PKV_SMEM_CASE(128, 8) PKV_SMEM_CASE(64, 1) PKV_SMEM_CASE(64, 2) PKV_SMEM_CASE(64, 4)
  PKV_SMEM_CASE(64, 6) PKV_SMEM_CASE(64, 8)
  if (per_warp == 0) return 0;
  return per_warp * kDecodeWarps + sizeof(int32_t) * (5 * (size_t)batch + 1);
}

cudaError_t launch_decode(const DecodeKernel& k, const DecodeArgs& a, int grid, size_t smem,
                          cudaStream_t stream) {
  DecodeArgs args = a;
  void* split_params[] = {&args};
  cudaError_t e = cudaLaunchKernel(k.split, dim3(grid), dim3(kDecodeWarps * 32), split_params, smem, stream);
  if (e != cudaSuccess) return e;
  int group = k.group;
  void* merge_params[] = {&args, &group};
  const int rows = a.B * a.Hq;
  const int mgrid = (rows + kMergeWarps - 1) / kMergeWarps;
  if (mgrid == 0) return cudaSuccess;
  return cudaLaunchKernel(k.merge, dim3(mgrid), dim3(kMergeWarps * 32), merge_params, 0, stream);
}

}  // namespace pkv
