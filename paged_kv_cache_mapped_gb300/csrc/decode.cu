// decode.cu -- single-token decode attention over a paged KV cache, for sm_103a.
//
// out[b,h] = softmax(scale * q[b,h] . K_t) . V_t over the attended tokens t of sequence b
// (the attention formula of "Transformer模型中的KV Cache优化推理策略", yutianautomatic.com,
// evaluated for one new query against the cached K/V as the KV-cache primer,
// cf-1.com/news/5988169, section 2.2 describes; K/V found through the block table of its
// section 4.1).  Dense mode attends [max(0, L-window), L); sparse mode attends a kept list
// (the layer-wise sparse variant of "How KV Sparsity Achieves 1.5x Acceleration for vLLM").
//
// Design (GB300-first; the step is HBM-bound at 4-6 flop per KV byte):
//  * Work partition (a "stream-K" split): the (sequence, kv head, 16-token unit) list is
//    flattened and cut into equal contiguous ranges, one per worker warp of a grid sized to
//    the SMs, so every worker streams the same number of bytes whatever the length mix.  A
//    range may end inside a (sequence, kv head) segment: each worker emits a partial
//    (running max m, running sum l, unnormalised o) per segment it touches, and a segment
//    covered by one worker writes its output directly.  A merge kernel combines the rest.
//  * Each worker warp owns a ring of K/V tile pairs in shared memory that complete on
//    per-slot mbarriers.  Dense mode fills them with TMA tiled copies of a 2-D tensor map
//    over the pool (one 64-column x 16-row box per 128 bytes of row, 128-byte swizzle, L2
//    evict-first): 4 copy operations per unit, and the swizzle puts the 8 rows an ldmatrix
//    reads in 8 different bank groups.  Sparse mode gathers rows: each lane issues one
//    256-byte cp.async.bulk row copy chosen through its kept index into rows stored at a
//    272-byte pitch (again conflict-free for ldmatrix).
//  * GQA: the G <= 8 query heads sharing a kv head are processed together, so each K/V byte
//    is read from HBM once per kv head.
//  * Both contractions run on the tensor cores as warp-level mma.m16n8k16 (bf16 inputs,
//    exact products, fp32 accumulation), with tokens as the 16-row dimension and heads as
//    the 8-column one: S^T = K q^T (16 tokens x 8 heads) and O^T += V^T P^T (d x 8 heads).
//    P^T leaves the first product as an accumulator fragment and becomes the second one's
//    operand by an in-register 8x8 transpose (movmatrix); it is carried as bf16 hi + lo
//    parts so P keeps ~16 significant bits.  This replaces ~870 CUDA-core instructions per
//    unit with ~100, leaving the warps waiting on memory rather than on issue slots.
//  * Online softmax ("How KV Sparsity...", section "2. Attention modification", Fig. 7:
//    running max, running sum, rescale, divide at the end) in base 2 with log2(e) folded
//    into the scale; the running max only moves when a unit's max exceeds it by 2^8, so the
//    output rescale is rare.
//  * Every wait is bounded (globaltimer); a timeout records PKV_DEV_WAIT_TIMEOUT, waits for
//    the copies in flight and returns.  Bad block ids / kept indices are skipped and
//    recorded, never dereferenced.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "pkv.h"

namespace pkv {
namespace {

template <int D, bool SPARSE>
struct Geo {
  static constexpr int kRow = D * 2;                       // bytes per K/V row in HBM
  static constexpr int kBoxes = D / 64;                    // dense: 128-byte column boxes per row
  static constexpr int kPitch = D * 2 + 16;                // sparse: padded row pitch in smem
  static constexpr int kTile = SPARSE ? 16 * kPitch : 16 * D * 2;  // bytes per 16-row tile
  static constexpr int kKSteps = D / 16;                   // k-steps of q.K, m-tiles of P.V
  static constexpr int kRing = (D == 128) ? PKV_RING_D128 : PKV_RING_D64;
  static_assert(kBoxes * 128 == kRow && kRing >= 2, "head_dim must be a multiple of 64");
};

// Byte offset inside a tile of the 16-byte chunk holding row r, columns [8c, 8c + 8).
// Dense tiles are kBoxes boxes of 16 rows x 128 bytes written by TMA with the 128-byte
// swizzle (chunk index XOR row % 8 inside each 1024-byte box); sparse tiles are plain rows
// at the padded pitch.
template <int D, bool SPARSE>
__device__ __forceinline__ uint32_t chunk_offset(int r, int c) {
  if constexpr (SPARSE) {
    return (uint32_t)(r * Geo<D, SPARSE>::kPitch + c * 16);
  } else {
    return (uint32_t)((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }
}

// A running max is only moved (and the output rescaled) when a unit's max exceeds it by more
// than this many base-2 units, so unnormalised weights stay below 2^8 and most units skip
// the rescale.  Any reference value gives the same normalised result.
constexpr float kRescaleSlack = 8.0f;

template <int D, bool SPARSE>
struct WarpTiles {
  alignas(1024) unsigned char k[Geo<D, SPARSE>::kRing][Geo<D, SPARSE>::kTile];
  alignas(1024) unsigned char v[Geo<D, SPARSE>::kRing][Geo<D, SPARSE>::kTile];
};

template <int D, bool SPARSE>
struct WarpSlots {
  uint64_t bar_k[Geo<D, SPARSE>::kRing];  // K rows of the slot landed
  uint64_t bar_v[Geo<D, SPARSE>::kRing];  // V rows of the slot landed
  uint32_t meta[Geo<D, SPARSE>::kRing];   // rows of the unit that were copied (bit t = token t)
  int32_t phys[Geo<D, SPARSE>::kRing];    // dense: physical block of the unit in the slot
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

template <int D, bool SPARSE>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  using GE = Geo<D, SPARSE>;
  using WT = WarpTiles<D, SPARSE>;
  using WB = WarpSlots<D, SPARSE>;
  constexpr int R = GE::kRing;
  constexpr int KS = GE::kKSteps;

  // Tile rings in static shared memory: the toolchain honours the 1 KiB alignment the
  // 128-byte swizzle pattern needs (it is a function of address bits 4-9).  The per-sequence
  // arrays, sized by the batch, are dynamic.
  static_assert((sizeof(WT) + sizeof(WB)) * kDecodeWarps <= 48 * 1024,
                "tile rings exceed static shared memory");
  __shared__ WT warps_tiles[kDecodeWarps];
  __shared__ WB warps_slots[kDecodeWarps];
  extern __shared__ __align__(16) int32_t smem_dyn[];
  int32_t* s_start = smem_dyn;
  int32_t* s_nb = s_start + (a.B + 1);
  int32_t* s_first = s_nb + a.B;
  int32_t* s_lo = s_first + a.B;   // dense: first attended token; sparse: context length
  int32_t* s_len = s_lo + a.B;     // dense: context length; sparse: kept count

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // fragment column pair
  const int G = a.G;
  WT& Wt = warps_tiles[warp];  // this warp's K/V tile ring
  WB& Wb = warps_slots[warp];  // its barriers and per-slot records

  if (lane == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(&Wb.bar_k[s], 1);
      mbar_init(&Wb.bar_v[s], 1);
    }
    fence_mbar_init();
  }
  // Launched with programmatic stream serialisation: wait for the previous kernel on the
  // stream before reading anything in global memory, then let the merge kernel launch.
  grid_dependency_wait();
  grid_launch_dependents();

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
  Cursor ic = locate(u0, s_start, s_nb, a.B);  // next unit to issue
  Cursor cc = ic;                               // next unit to consume

  // q of the next segment as raw bf16x2 words in B-fragment order: word 2ks+i holds head gq's
  // elements 16ks + 8i + 2tq, +1 (zero for heads >= G).  The first segment's right away.
  uint32_t qraw[2 * KS];
  auto load_q = [&](int b, int g) {
    if (gq < G) {
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + (size_t)g * G + gq) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qraw[2 * ks] = __ldg(qw + ks * 8 + tq);
        qraw[2 * ks + 1] = __ldg(qw + ks * 8 + 4 + tq);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2 * KS; ++i) qraw[i] = 0u;
    }
  };
  load_q(cc.b, cc.g);

  // Dense: the block-table entries of this worker's units, 32 per coalesced load (lane l
  // holds the entry of unit chunk_base + l), fetched one chunk ahead of use.
  int bt_cur = -1, bt_next = -1, chunk_base = 0;
  auto load_chunk = [&](int first) -> int {
    int phys = -1;
    if (first + lane < nunits) {
      const Cursor c = locate(u0 + first + lane, s_start, s_nb, a.B);
      phys = __ldg(a.block_tables + (size_t)c.b * a.MB + s_first[c.b] + c.j);
    }
    return phys;
  };
  if constexpr (!SPARSE) {
    bt_cur = load_chunk(0);
    if (nunits > 32) bt_next = load_chunk(32);
  }

  // Issue unit k (the one `ic` names) into slot k % R.  Dense: lane 0 copies the K and V
  // tiles as TMA boxes.  Sparse: lane r < 16 copies K row r, lane 16 + r V row r.
  auto issue = [&](int k) {
    const int slot = k % R;
    fence_proxy_async_smem();
    if constexpr (!SPARSE) {
      if (k - chunk_base == 32) {
        chunk_base += 32;
        bt_cur = bt_next;
        if (chunk_base + 32 < nunits) bt_next = load_chunk(chunk_base + 32);
      }
      const int phys = __shfl_sync(kFullMask, bt_cur, k - chunk_base);
      if (lane == 0) {
        if (phys >= 0 && phys < a.NB) {
          const int y = (phys * a.Hkv + ic.g) * 16;  // host checks NB*Hkv*16 < 2^31
          Wb.meta[slot] = 0xffffu;
          Wb.phys[slot] = phys;
          mbar_arrive_expect_tx(&Wb.bar_k[slot], GE::kTile);
#pragma unroll
          for (int bx = 0; bx < GE::kBoxes; ++bx)
            tma_load_2d(Wt.k[slot] + bx * 2048, &a.tmap_k, bx * 64, y, &Wb.bar_k[slot], pol);
          mbar_arrive_expect_tx(&Wb.bar_v[slot], GE::kTile);
#pragma unroll
          for (int bx = 0; bx < GE::kBoxes; ++bx)
            tma_load_2d(Wt.v[slot] + bx * 2048, &a.tmap_v, bx * 64, y, &Wb.bar_v[slot], pol);
        } else {
          record_error(a.err, PKV_DEV_BAD_BLOCK_ID);
          Wb.meta[slot] = 0u;
          mbar_arrive_expect_tx(&Wb.bar_k[slot], 0);
          mbar_arrive_expect_tx(&Wb.bar_v[slot], 0);
        }
      }
      advance(ic, s_nb, a.B, a.Hkv);
    } else {
      const int r = lane & 15;
      const bool is_v = lane >= 16;
      bool ok;
      size_t src = 0;
      const int pos = ic.j * 16 + r;
      ok = pos < s_len[ic.b];
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
      src = (((size_t)phys * a.Hkv + ic.g) * 16 + (t & 15)) * D;
      const uint32_t vmask = __ballot_sync(kFullMask, ok) & 0xffffu;  // K and V lanes agree
      if (lane == 0) {
        Wb.meta[slot] = vmask;
        mbar_arrive_expect_tx(&Wb.bar_k[slot], __popc(vmask) * GE::kRow);
        mbar_arrive_expect_tx(&Wb.bar_v[slot], __popc(vmask) * GE::kRow);
      }
      __syncwarp();
      if (ok) {
        unsigned char* dst = (is_v ? Wt.v[slot] : Wt.k[slot]) + r * GE::kPitch;
        bulk_g2s(dst, (is_v ? a.v_cache : a.k_cache) + src, GE::kRow, is_v ? &Wb.bar_v[slot] : &Wb.bar_k[slot], pol);
      }
      advance(ic, s_nb, a.B, a.Hkv);
    }
  };

  int issued = 0;
  for (; issued < nunits && issued < R; ++issued) issue(issued);

  // ---- consumer state: this lane's heads are h0 = 2tq and h1 = 2tq + 1 ------------------
  uint32_t qb[2 * KS];   // q^T B fragments of the current segment
  float o[KS][4];        // O^T accumulator fragments: [m-tile][d row gq / gq+8, head h0 / h1]
  float mr0 = -INFINITY, mr1 = -INFINITY;  // running max (reference) of heads h0, h1
  float l0 = 0.f, l1 = 0.f;                // this lane's share of the running sums
  int seg_b = -1, seg_g = -1, part = 0, nparts = 0;
  const float sl2 = a.scale_log2;
  // Dense append mode: this step's K (lanes 0-15) or V (lanes 16-31) row chunk of the current
  // segment, to be written at token L_b - 1 (pool and tile) when its unit is consumed.
  const bool appending = !SPARSE && a.k_new != nullptr;
  uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
  const int new_chunk = lane & 15;
  const bool new_lane = new_chunk < D / 8;

  auto flush = [&]() {
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
      l0 += __shfl_xor_sync(kFullMask, l0, m);
      l1 += __shfl_xor_sync(kFullMask, l1, m);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int head = 2 * tq + hh;
      if (head >= G) continue;
      const float l = hh ? l1 : l0;
      const float m = hh ? mr1 : mr0;
      const size_t row = (size_t)seg_b * a.Hq + (size_t)seg_g * G + head;
      if (nparts == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* dst = a.out + row * D + gq;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          dst[mt * 16] = __float2bfloat16_rn(o[mt][hh] * inv);
          dst[mt * 16 + 8] = __float2bfloat16_rn(o[mt][2 + hh] * inv);
        }
      } else {
        float* dst = a.part_o + (row * a.max_parts + part) * D + gq;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          dst[mt * 16] = o[mt][hh];
          dst[mt * 16 + 8] = o[mt][2 + hh];
        }
        if (gq == 0) a.part_ml[row * a.max_parts + part] = make_float2(m, l);
      }
    }
  };

  auto begin_segment = [&](const Cursor& c) {
    seg_b = c.b;
    seg_g = c.g;
    const int nb = s_nb[c.b];
    const int seg_begin = s_start[c.b] + c.g * nb;
    const int w0 = seg_begin / per;
    nparts = (seg_begin + nb - 1) / per - w0 + 1;
    part = (int)gw - w0;
#pragma unroll
    for (int i = 0; i < 2 * KS; ++i) qb[i] = qraw[i];
    if (appending && new_lane) {
      const __nv_bfloat16* src = (lane >= 16 ? a.v_new : a.k_new) + ((size_t)c.b * a.Hkv + c.g) * D + new_chunk * 8;
      new_row = __ldg(reinterpret_cast<const uint4*>(src));
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;
    mr0 = mr1 = -INFINITY;
    l0 = l1 = 0.f;
    // prefetch q of the segment that follows, if this worker reaches it
    if (seg_begin + nb < u0 + nunits) {
      int nb2 = c.b, ng2 = c.g + 1;
      if (ng2 == a.Hkv) {
        ng2 = 0;
        do { ++nb2; } while (nb2 < a.B && s_nb[nb2] == 0);
      }
      if (nb2 < a.B) load_q(nb2, ng2);
    }
  };

  // ldmatrix rows of this lane: K (non-transposed A of S^T = K q^T) reads row lane & 15, chunk
  // 2 ks + lane / 16; V (transposed A of O^T = V^T P^T) reads token (lane & 7) + 8 (lane / 16),
  // chunk 2 mt + (lane / 8) % 2.
  const int k_row = lane & 15, k_half = lane >> 4;
  const int v_row = (lane & 7) + ((lane >> 4) << 3), v_half = (lane >> 3) & 1;

  bool aborted = false;
  int k = 0;
  for (; k < nunits; ++k) {
    if (cc.b != seg_b || cc.g != seg_g) {
      if (seg_b >= 0) flush();
      begin_segment(cc);
    }
    const int slot = k % R;
    const uint32_t parity = (uint32_t)(k / R) & 1u;
    // every lane waits (acquiring the TMA writes); the give-up decision is warp-uniform
    if (!__all_sync(kFullMask, mbar_wait_bounded(&Wb.bar_k[slot], parity, a.timeout_ns))) {
      if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    uint32_t mask = Wb.meta[slot];
    int t_new = -1;  // tile row of this step's token when the unit holds it (append mode)
    if constexpr (!SPARSE) {
      const int tok0 = (s_first[cc.b] + cc.j) * 16;
      const int lo = max(s_lo[cc.b] - tok0, 0);
      const int hi = min(s_len[cc.b] - tok0, 16);
      mask &= ((1u << hi) - 1u) & ~((1u << lo) - 1u);
      if (appending && mask != 0u && s_len[cc.b] - 1 - tok0 < 16) {
        t_new = s_len[cc.b] - 1 - tok0;
        // the tile was read before the append: put the new K row in it and in the pool
        if (lane < 16 && new_lane) {
          *reinterpret_cast<uint4*>(Wt.k[slot] + chunk_offset<D, SPARSE>(t_new, new_chunk)) = new_row;
          *reinterpret_cast<uint4*>(a.k_pool_out + (((size_t)Wb.phys[slot] * a.Hkv + cc.g) * 16 + t_new) * D +
                                    new_chunk * 8) = new_row;
        }
        __syncwarp();
      }
    }
    if (mask != 0u) {
      // -- S^T = K q^T: 16 tokens x 8 heads --------------------------------------------------
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t kbase = smem_u32(Wt.k[slot]);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t af[4];
        ldsm_x4(kbase + chunk_offset<D, SPARSE>(k_row, 2 * ks + k_half), af);
        mma_bf16_m16n8k16(c, af, qb[2 * ks], qb[2 * ks + 1]);
      }
      // c[0] = (token gq, head h0), c[1] = (gq, h1), c[2] = (gq + 8, h0), c[3] = (gq + 8, h1)
      const bool t0 = (mask >> gq) & 1u;
      const bool t1 = (mask >> (gq + 8)) & 1u;
      const bool v0 = 2 * tq < G, v1 = 2 * tq + 1 < G;
      const float s00 = (t0 && v0) ? c[0] * sl2 : -INFINITY;
      const float s01 = (t0 && v1) ? c[1] * sl2 : -INFINITY;
      const float s10 = (t1 && v0) ? c[2] * sl2 : -INFINITY;
      const float s11 = (t1 && v1) ? c[3] * sl2 : -INFINITY;
      float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, m));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, m));
      }
      // lazy running max: move it only when this unit's max is well above it
      const bool g0 = mx0 > mr0 + kRescaleSlack, g1 = mx1 > mr1 + kRescaleSlack;
      if (__any_sync(kFullMask, g0 || g1)) {
        float al0 = 1.f, al1 = 1.f;
        if (g0) {
          al0 = exp2f(mr0 - mx0);
          mr0 = mx0;
        }
        if (g1) {
          al1 = exp2f(mr1 - mx1);
          mr1 = mx1;
        }
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
      }
      const float ref0 = (mr0 == -INFINITY) ? 0.f : mr0;
      const float ref1 = (mr1 == -INFINITY) ? 0.f : mr1;
      const float p00 = exp2f(s00 - ref0), p01 = exp2f(s01 - ref1);
      const float p10 = exp2f(s10 - ref0), p11 = exp2f(s11 - ref1);
      l0 += p00 + p10;
      l1 += p01 + p11;
      // -- P^T as bf16 hi + lo B fragments (tokens x heads -> heads x tokens) -------------
      const uint32_t hA = pack_bf16x2(p00, p01);  // token gq
      const uint32_t hB = pack_bf16x2(p10, p11);  // token gq + 8
      const uint32_t lA = pack_bf16x2(p00 - bf16_lo_to_f32(hA), p01 - bf16_hi_to_f32(hA));
      const uint32_t lB = pack_bf16x2(p10 - bf16_lo_to_f32(hB), p11 - bf16_hi_to_f32(hB));
      const uint32_t bh0 = movmatrix_trans(hA), bh1 = movmatrix_trans(hB);
      const uint32_t bl0 = movmatrix_trans(lA), bl1 = movmatrix_trans(lB);
      if (!__all_sync(kFullMask, mbar_wait_bounded(&Wb.bar_v[slot], parity, a.timeout_ns))) {
        if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
        break;
      }
      if (t_new >= 0) {  // append mode: the new V row, into the tile and the pool
        if (lane >= 16 && new_lane) {
          *reinterpret_cast<uint4*>(Wt.v[slot] + chunk_offset<D, SPARSE>(t_new, new_chunk)) = new_row;
          *reinterpret_cast<uint4*>(a.v_pool_out + (((size_t)Wb.phys[slot] * a.Hkv + cc.g) * 16 + t_new) * D +
                                    new_chunk * 8) = new_row;
        }
        __syncwarp();
      }
      if (mask != 0xffffu) {
        // rows of tokens outside the attended set may hold anything (even NaN): zero them,
        // since the tensor core would turn 0 * NaN into NaN
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 2 * i + (lane >> 4);
          const int c = lane & 15;  // chunk (16 bytes) of the row
          if (!((mask >> t) & 1u) && c < D / 8)
            *reinterpret_cast<uint4*>(Wt.v[slot] + chunk_offset<D, SPARSE>(t, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      // -- O^T += V^T P^T -------------------------------------------------------------------
      const uint32_t vbase = smem_u32(Wt.v[slot]);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t av[4];
        ldsm_x4_trans(vbase + chunk_offset<D, SPARSE>(v_row, 2 * mt + v_half), av);
        mma_bf16_m16n8k16(o[mt], av, bh0, bh1);
        mma_bf16_m16n8k16(o[mt], av, bl0, bl1);
      }
    } else if (!__all_sync(kFullMask, mbar_wait_bounded(&Wb.bar_v[slot], parity, a.timeout_ns))) {
      if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    __syncwarp();
    if (issued < nunits) {
      issue(issued);
      ++issued;
    }
    advance(cc, s_nb, a.B, a.Hkv);
  }

  if (aborted) {  // let the copies in flight land before the CTA's shared memory goes away
    for (int kk = k; kk < issued; ++kk) {
      (void)mbar_wait_bounded(&Wb.bar_k[kk % R], (uint32_t)(kk / R) & 1u, a.timeout_ns);
      (void)mbar_wait_bounded(&Wb.bar_v[kk % R], (uint32_t)(kk / R) & 1u, a.timeout_ns);
    }
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
  grid_dependency_wait();  // the split kernel's partials and partition record
  grid_launch_dependents();
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
  // Partials in groups of 32: lane p holds (m, l) of partial p; the o loads of a group are
  // independent of the weights, so one memory round trip covers a group.
  float M = -INFINITY, L = 0.f;
  float acc[EPW];
#pragma unroll
  for (int e = 0; e < EPW; ++e) acc[e] = 0.f;
  for (int p0 = 0; p0 < np; p0 += 32) {
    const int n = min(32, np - p0);
    const float2 mlp = lane < n ? __ldcg(ml + p0 + lane) : make_float2(-INFINITY, 0.f);
    float gmax = mlp.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(kFullMask, gmax, o));
    const float M_new = fmaxf(M, gmax);
    const float mref = (M_new == -INFINITY) ? 0.f : M_new;
    const float carry = exp2f(M - mref);  // rescale what earlier groups accumulated
    L *= carry;
#pragma unroll
    for (int e = 0; e < EPW; ++e) acc[e] *= carry;
    M = M_new;
    const float w_lane = exp2f(mlp.x - mref);
    float lsum = w_lane * mlp.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(kFullMask, lsum, o);
    L += lsum;
    // batches of 8 partials: all loads of a batch are issued before any is used
    for (int pb = 0; pb < n; pb += 8) {
      float x[8][EPW];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (pb + j < n) {
          const float* src = po + (size_t)(p0 + pb + j) * D;
          if constexpr (EPW == 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
            x[j][0] = v.x; x[j][1] = v.y; x[j][2] = v.z; x[j][3] = v.w;
          } else {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
            x[j][0] = v.x; x[j][1] = v.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = __shfl_sync(kFullMask, w_lane, (pb + j) & 31);
        if (pb + j < n) {
#pragma unroll
          for (int e = 0; e < EPW; ++e) acc[e] += w * x[j][e];
        }
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < EPW; e += 2) {
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

}  // namespace

DecodeKernel decode_kernel(int head_dim, int group, bool sparse) {
  if (group < 1 || group > kMaxGroup) return DecodeKernel{nullptr, nullptr, head_dim, group, sparse};
  if (head_dim == 128)
    return DecodeKernel{sparse ? (const void*)decode_split_kernel<128, true>
                               : (const void*)decode_split_kernel<128, false>,
                        (const void*)decode_merge_kernel<128>, 128, group, sparse};
  if (head_dim == 64)
    return DecodeKernel{sparse ? (const void*)decode_split_kernel<64, true>
                               : (const void*)decode_split_kernel<64, false>,
                        (const void*)decode_merge_kernel<64>, 64, group, sparse};
  return DecodeKernel{nullptr, nullptr, head_dim, group, sparse};
}

size_t decode_smem_bytes(int head_dim, bool sparse, int batch) {
  (void)sparse;
  if (head_dim != 128 && head_dim != 64) return 0;
  // dynamic part only: the per-sequence arrays (the tile rings are static)
  return sizeof(int32_t) * (5 * (size_t)batch + 1);
}

cudaError_t launch_decode(const DecodeKernel& k, const DecodeArgs& a, int grid, size_t smem,
                          cudaStream_t stream) {
  DecodeArgs args = a;
  args.G = k.group;
  void* split_params[] = {&args};
  cudaError_t e = launch_pdl(k.split, dim3(grid), dim3(kDecodeWarps * 32), smem, stream, split_params);
  if (e != cudaSuccess) return e;
  int group = k.group;
  void* merge_params[] = {&args, &group};
  const int rows = a.B * a.Hq;
  const int mgrid = (rows + kMergeWarps - 1) / kMergeWarps;
  if (mgrid == 0) return cudaSuccess;
  return launch_pdl(k.merge, dim3(mgrid), dim3(kMergeWarps * 32), 0, stream, merge_params);
}

}  // namespace pkv
