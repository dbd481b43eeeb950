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
//  * Work partition (a "stream-K" split with a dynamic tail): the (sequence, kv head,
//    16-token unit) list is flattened and cut into one equal slice per worker warp of a grid
//    sized to the SMs, so every worker streams about the same number of bytes whatever the
//    length mix.  A slice is a static head, run by the warp of the same index, and a few tail
//    chunks of halving length that warps take from a ticket counter once their own work is
//    done: warps on SMs that stream faster (SMs differ by up to ~20% in sustained bandwidth)
//    absorb the work of slower ones, which shortens the end of the launch.  A range (a head
//    or a chunk) may start or end inside a (sequence, kv head) segment: it then emits a
//    partial (running max m, running sum l, unnormalised o) into slots fixed by the range,
//    so the result does not depend on which warp ran it; a segment inside one range is
//    written out directly.  A merge kernel combines the partials.
//  * Each worker warp owns a ring of K/V tile pairs in shared memory that complete on
//    per-slot mbarriers.  Dense mode fills them with TMA tiled copies of a 2-D tensor map
//    over the pool (one 64-column x 16-row box per 128 bytes of row, 128-byte swizzle, L2
//    evict-first): 4 copy operations per unit, and the swizzle puts the 8 rows an ldmatrix
//    reads in 8 different bank groups.  Sparse mode gathers rows chosen through their kept
//    indices as 16-byte cp.async chunks (each lane one chunk of several rows) into the same
//    swizzled layout, so both modes share the consumer.
//  * GQA: the G <= 8 query heads sharing a kv head are processed together, so each K/V byte
//    is read from HBM once per kv head.
//  * Both contractions run on the tensor cores as warp-level mma.m16n8k16 (bf16 inputs,
//    exact products, fp32 accumulation), with tokens as the 16-row dimension and heads as
//    the 8-column one: S^T = K q^T (16 tokens x 8 heads) and O^T += V^T P^T (d x 8 heads).
//    P^T leaves the first product as an accumulator fragment and becomes the second one's
//    operand by an in-register 8x8 transpose (movmatrix); it is carried as bf16 hi + lo
//    parts so P keeps ~16 significant bits.  This replaces ~870 CUDA-core instructions per
//    unit with ~100, leaving the warps waiting on memory rather than on issue slots.
//  * INT8 pools (one byte per element, the code + 128, plus one fp32 scale per row and kv
//    head): the codes become fp16 in registers (a byte permute under the exponent of 1024,
//    and for V one subtraction per pair), both products take fp16 operands, the K row scales multiply the
//    logits and the V row scales enter P, relative to a per-segment reference scale, as one
//    fp16 term.  Sparse rows arrive chunk by chunk as above, their scales as 4-byte copies
//    completing on the K barrier.
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

// Q8: INT8 pools, one byte per element; a tile is a single TMA box of 16 rows x D bytes.
template <int D, bool SPARSE, bool Q8 = false>
struct Geo {
  static constexpr int kRow = Q8 ? D : D * 2;              // bytes per K/V row in HBM
  static constexpr int kBoxes = Q8 ? 1 : D / 64;           // dense: 128-byte column boxes per row
  static constexpr int kTile = 16 * kRow;                  // bytes per tile
  static constexpr int kKSteps = D / 16;                   // k-steps of q.K, m-tiles of P.V
  static constexpr int kRing = (SPARSE && D == 128) ? PKV_RING_SPARSE_D128
                               : Q8 ? ((D == 128) ? PKV_RING_Q8_D128 : PKV_RING_Q8_D64)
                                    : ((D == 128) ? PKV_RING_D128 : PKV_RING_D64);
  static_assert((Q8 || kBoxes * 128 == kRow) && kRing >= 2, "head_dim must be a multiple of 64");
};

// Byte offset inside a tile of the 16-byte chunk c of row r.
// bf16 tiles are kBoxes boxes of 16 rows x 128 bytes, in the layout TMA writes with the 128-byte
// swizzle (chunk index XOR row % 8 inside each 1024-byte box).
// INT8 tiles are one box of 16 rows x D bytes, in the layout of the swizzle of the row size:
// 128 bytes (chunk XOR row % 8) at D = 128, 64 bytes (chunk XOR (row / 2) % 4) at D = 64.
// Either way the 8 rows an ldmatrix reads land in 8 different bank groups.  The gather form
// writes the same layout chunk by chunk (cp.async), so both forms share one consumer.
template <int D, bool SPARSE, bool Q8 = false>
__device__ __forceinline__ uint32_t chunk_offset(int r, int c) {
  if constexpr (Q8) {
    if constexpr (D == 128)
      return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
    else
      return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
  } else {
    return (uint32_t)((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }
}

// A running max is only moved (and the output rescaled) when a unit's max exceeds it by more
// than this many base-2 units, so unnormalised weights stay below 2^8 and most units skip
// the rescale.  Any reference value gives the same normalised result.
constexpr float kRescaleSlack = 8.0f;
// INT8 pools: the V-scale reference moves when a unit's largest V scale exceeds it by this
// factor, so P times scale / reference stays below 2^8 * 64 (inside fp16).
constexpr float kVrefSlack = 64.0f;

template <int D, bool SPARSE, bool Q8 = false>
struct WarpTiles {
  alignas(1024) unsigned char k[Geo<D, SPARSE, Q8>::kRing][Geo<D, SPARSE, Q8>::kTile];
  alignas(1024) unsigned char v[Geo<D, SPARSE, Q8>::kRing][Geo<D, SPARSE, Q8>::kTile];
};

template <int D, bool SPARSE, bool Q8 = false>
struct WarpSlots {
  uint64_t bar_k[Geo<D, SPARSE, Q8>::kRing];  // K rows of the slot landed
  uint64_t bar_v[Geo<D, SPARSE, Q8>::kRing];  // V rows of the slot landed
  uint32_t meta[Geo<D, SPARSE, Q8>::kRing];   // rows of the unit that were copied (bit t = token t)
  int32_t phys[Geo<D, SPARSE, Q8>::kRing];    // dense: physical block of the unit in the slot
};

// INT8 pools: the row scales of the K and V tiles of each slot, copied with the K tile.
template <int R>
struct WarpScales {
  alignas(16) float k[R][16];
  alignas(16) float v[R][16];
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

// ---- the partition of the unit list into ranges ------------------------------------------
// p is the partition record (PartField).  Slice w covers units [wP, (w+1)P).  A full slice is
// its static head [wP, wP+S) followed by cpw tail chunks: chunk c covers
// [wP+S+O_c, wP+S+O_{c+1}) of a tail of T = P - S units, with O_c = T - floor(T (2^(cpw-c) - 1)
// / (2^cpw - 1)), so chunk lengths halve from one to the next.  Tickets hand out every slice's
// chunk c before any chunk c+1: the long chunks go first and the short ones even out the end
// (guided self-scheduling).  A partial last slice is one static range ending at the total.
// Every chunk is at least as long as a worker's tile ring.
//
// A range is named by rid = (w << kRangeShift) | j, j = 0 for the head and c + 1 for chunk c,
// so no division recovers its slice; range_index(rid) = w (1 + cpw) + j numbers the ranges in
// unit order (it indexes the partial slots).
constexpr int kRangeShift = 3;

__device__ __forceinline__ int range_of(const int32_t* p, int u) {
  const int P = p[kPartP], S = p[kPartS];
  const int w = u / P, o = u - w * P;
  if (o < S || w >= p[kPartNfull]) return w << kRangeShift;
  const int cpw = p[kPartCpw], ot = o - S;
  int c = 0;
  while (c + 1 < cpw && p[kPartOff + c + 1] <= ot) ++c;
  return (w << kRangeShift) | (c + 1);
}

__device__ __forceinline__ int range_start(const int32_t* p, int rid) {
  const int w = rid >> kRangeShift, j = rid & ((1 << kRangeShift) - 1);
  return w * p[kPartP] + (j == 0 ? 0 : p[kPartS] + p[kPartOff + j - 1]);
}

__device__ __forceinline__ int range_end(const int32_t* p, int rid) {
  const int w = rid >> kRangeShift, j = rid & ((1 << kRangeShift) - 1);
  if (w >= p[kPartNfull]) return p[kPartTotal];
  return w * p[kPartP] + p[kPartS] + (j == 0 ? 0 : p[kPartOff + j]);
}

__device__ __forceinline__ int range_index(const int32_t* p, int rid) {
  return (rid >> kRangeShift) * (1 + p[kPartCpw]) + (rid & ((1 << kRangeShift) - 1));
}

// The range of tail ticket t < p[kPartTickets]: chunk t / nfull of slice t % nfull.
__device__ __forceinline__ int ticket_range(const int32_t* p, int t) {
  const int nfull = p[kPartNfull];
  const int c = t / nfull;
  return ((t - c * nfull) << kRangeShift) | (c + 1);
}

constexpr uint32_t kNoTicket = 0xffffffffu;



// Batches up to this size let the merge kernel derive its rows' partitions from the lengths
// before the split kernel ends; larger ones read the split kernel's record after it.
constexpr int kMergeScanMaxBatch = 256;

// Units (16-token blocks of one kv head) that sequence b attends, with the bounds the split
// kernel needs; invalid lengths count as empty and return the device error to report.
struct SeqUnits {
  int nb;     // units
  int first;  // dense: first attended block; sparse: 0
  int lo;     // dense: first attended token; sparse: context length
  int len;    // dense: context length; sparse: kept count
  int err;    // PKV_DEV_* code or 0
};

template <bool SPARSE>
__device__ __forceinline__ SeqUnits seq_units(const DecodeArgs& a, int b) {
  SeqUnits s{0, 0, 0, 0, 0};
  int L = a.context_lens[b];
  if (L < 0 || L > a.MB * 16) {
    s.err = PKV_DEV_BAD_CONTEXT_LEN;
    L = 0;
  }
  if constexpr (SPARSE) {
    int n = a.kept_lens[b];
    if (n < 0 || n > a.max_kept) {
      if (s.err == 0) s.err = PKV_DEV_BAD_KEPT_INDEX;
      n = 0;
    }
    s.nb = (n + 15) >> 4;
    s.lo = L;
    s.len = n;
  } else {
    s.lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
    s.first = s.lo >> 4;
    s.nb = L > 0 ? ((L - 1) >> 4) - s.first + 1 : 0;
    s.len = L;
  }
  return s;
}

// Partition of `total` units over `nw` worker warps (total < 2^30).
__device__ void make_partition(int32_t* p, int total, int nw, const DecodeArgs& a) {
  int P = (total + nw - 1) / nw;
  // a slice of at least min_units, unless that would leave fewer than min_busy_pct % of the
  // workers with a slice
  const int busy = max(1, (int)((long long)nw * a.min_busy_pct / 100));
  const int floor_units = min(a.min_units, (total + busy - 1) / busy);
  if (P < floor_units) P = floor_units;
  // as many halving chunks as keep the last one, floor(T / (2^cpw - 1)), >= chunk_min
  const int tail = (int)((long long)P * a.tail_pct / 100);
  int cpw = 0;
  while (cpw < a.cpw_cap && tail >= a.chunk_min * ((2 << cpw) - 1)) ++cpw;
  const int T = cpw > 0 ? tail : 0;
  const int nfull = total / P;
  p[kPartTotal] = total;
  p[kPartP] = P;
  p[kPartS] = P - T;
  p[kPartTail] = T;
  p[kPartCpw] = cpw;
  p[kPartNfull] = nfull;
  p[kPartTickets] = nfull * cpw;
  p[kPartWorkers] = nfull + (nfull * P < total ? 1 : 0);
  for (int c = 0; c <= cpw; ++c)
    p[kPartOff + c] = cpw > 0 ? T - (int)((long long)T * ((1 << (cpw - c)) - 1) / ((1 << cpw) - 1)) : 0;
}

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// SCORES (dense only): also keep every attended key's base-2 logit and write the log-sum-exp of
// rows written out directly, for the score step (decode_score_kernel).
template <int D, bool SPARSE, bool SCORES, bool Q8>
__global__ void __launch_bounds__(kDecodeWarps * 32, Q8 ? PKV_Q8_MIN_CTAS : 0)
decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  static_assert(!(SPARSE && SCORES), "scores are emitted by the dense decode only");
  using GE = Geo<D, SPARSE, Q8>;
  using WT = WarpTiles<D, SPARSE, Q8>;
  using WB = WarpSlots<D, SPARSE, Q8>;
  constexpr int R = GE::kRing;
  constexpr int KS = GE::kKSteps;

  // Tile rings in static shared memory: the toolchain honours the 1 KiB alignment the
  // 128-byte swizzle pattern needs (it is a function of address bits 4-9).  The per-sequence
  // arrays, sized by the batch, are dynamic.
  static_assert((sizeof(WT) + sizeof(WB)) * kDecodeWarps <= 48 * 1024,
                "tile rings exceed static shared memory");
  __shared__ WT warps_tiles[kDecodeWarps];
  __shared__ WB warps_slots[kDecodeWarps];
  __shared__ WarpScales<Q8 ? GE::kRing : 1> warps_scales[Q8 ? kDecodeWarps : 1];  // INT8 pools only
  __shared__ int32_t s_part[kPartFields];
  __shared__ uint32_t s_ticket[kDecodeWarps];
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
  // Launched with programmatic stream serialisation: the previous kernel on the stream may
  // still run.  Normally the kernel waits for it before reading anything in global memory.
  // With a.early the caller has declared the pools, block tables, lengths and kept lists final
  // before that kernel: the partition, the first range's table entries and its first ring of
  // tile copies go ahead, and the wait comes before the first read of q, the new rows or the
  // workspace (and before the first error-word write: errors found earlier are held in
  // `pending_err`).  The merge kernel may launch once this kernel has waited, so at most the
  // previous call's kernels run alongside an early prologue.
  bool waited = a.early == 0;
  int pending_err = 0;
  if (waited) {
    grid_dependency_wait();
    grid_launch_dependents();
  }
  auto note_error = [&](int code) {
    if (waited) record_error(a.err, code);
    else if (pending_err == 0) pending_err = code;
  };

  // ---- per-sequence unit counts and partition (identical in every CTA) -------------------
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const SeqUnits su = seq_units<SPARSE>(a, b);
    if (su.err != 0 && blockIdx.x == 0) note_error(su.err);
    if constexpr (SCORES) {  // a context longer than the score rows: its keys beyond them get no score
      if (su.len > a.score_stride && blockIdx.x == 0) note_error(PKV_DEV_BAD_CONTEXT_LEN);
    }
    s_nb[b] = su.nb;
    s_first[b] = su.first;
    s_lo[b] = su.lo;
    s_len[b] = su.len;
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
    if (lane == 0) {
      s_start[a.B] = carry;
      make_partition(s_part, carry, a.workers, a);
    }
  }
  __syncthreads();

  // Large batches: the merge kernel reads the unit starts from here rather than recomputing
  // them (smaller ones it derives from the lengths while this kernel still runs).  The record
  // is in the workspace, so it is written once the previous kernel has ended.
  auto write_layout = [&]() {
    if (blockIdx.x == 0 && a.B > kMergeScanMaxBatch) {
      for (int i = threadIdx.x; i < a.B; i += blockDim.x) a.layout[i] = s_start[i];
      for (int i = threadIdx.x; i < a.B; i += blockDim.x) a.layout[a.B + i] = s_nb[i];
    }
  };
  // the early prologue's end: wait for the previous kernel, let the merge launch, then the
  // writes held back
  auto finish_wait = [&]() {
    if (waited) return;
    grid_dependency_wait();
    grid_launch_dependents();
    waited = true;
    if (pending_err != 0) record_error(a.err, pending_err);
    write_layout();
  };
  if (waited) write_layout();
  const int gw = (int)blockIdx.x * kDecodeWarps + warp;
  const int tickets = s_part[kPartTickets];
  uint32_t n_taken = 0;        // tail tickets this warp took
  uint32_t t_req = kNoTicket;  // lane 0: a ticket requested before the current range ends
  // The next range from the ticket counter, or -1 (lane 0 hands the ticket over through
  // shared memory, so every lane sees the same value).
  auto take_ticket = [&]() -> int {
    int r = -1;
    if (tickets > 0) {
      if (lane == 0) s_ticket[warp] = (t_req == kNoTicket) ? atomicAdd(a.ctrl, 1u) : t_req;
      t_req = kNoTicket;
      __syncwarp();
      const uint32_t t = s_ticket[warp];
      __syncwarp();
      if (t < (uint32_t)tickets) {
        ++n_taken;
        r = ticket_range(s_part, (int)t);
      }
    }
    return r;
  };
  // this warp's first range: its slice's static head, or a tail chunk
  int rid = gw << kRangeShift;
  if (gw >= s_part[kPartWorkers]) {
    finish_wait();  // the ticket counter is in the workspace
    rid = take_ticket();
  }
  bool aborted = false;
  bool first_range = true;
  while (rid >= 0 && !aborted) {
  const int u0 = range_start(s_part, rid);
  const int nunits = range_end(s_part, rid) - u0;
  const int ridx = range_index(s_part, rid);
  if (!first_range) {
    // a new range restarts the tile ring from phase 0 (every copy of the last one has landed)
    __syncwarp();
    if (lane == 0) {
      for (int s = 0; s < R; ++s) {
        mbar_inval(&Wb.bar_k[s]);
        mbar_inval(&Wb.bar_v[s]);
        mbar_init(&Wb.bar_k[s], 1);
        mbar_init(&Wb.bar_v[s], 1);
      }
      fence_mbar_init();
    }
    __syncwarp();
  }
  first_range = false;

  const uint64_t pol = l2_policy_evict_first();
  Cursor ic = locate(u0, s_start, s_nb, a.B);  // next unit to issue
  Cursor cc = ic;                               // next unit to consume

  // q of the next segment as raw bf16x2 words in B-fragment order: word 2ks+i holds head gq's
  // elements 16ks + 8i + 2tq, +1 (zero for heads >= G).  The first segment's right away.
  // INT8 pools: word 2ks+i holds elements 16ks + 4tq + 2i, +1 (the order in which an ldmatrix
  // of int8 rows hands each lane its K bytes: four consecutive columns).
  uint32_t qraw[2 * KS];
  auto load_q = [&](int b, int g) {
    if (gq < G) {
      if constexpr (Q8) {
        const uint2* qw = reinterpret_cast<const uint2*>(a.q + ((size_t)b * a.Hq + (size_t)g * G + gq) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint2 w = __ldg(qw + ks * 4 + tq);
          qraw[2 * ks] = w.x;
          qraw[2 * ks + 1] = w.y;
        }
      } else {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + (size_t)g * G + gq) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qraw[2 * ks] = __ldg(qw + ks * 8 + tq);
          qraw[2 * ks + 1] = __ldg(qw + ks * 8 + 4 + tq);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2 * KS; ++i) qraw[i] = 0u;
    }
  };
  if (waited) load_q(cc.b, cc.g);

  // Dense: the block-table entries of this range's units, 32 per coalesced load (lane l
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
  // Sparse: the rows of this range's units are resolved in pairs of units (lane l: slot l & 15
  // of unit 2c + l / 16) through a pipeline -- the kept entry two pairs ahead of issue, its block
  // id one pair ahead, the pool row at issue -- so an issue waits on neither dependent load.  An
  // entry outside [0, L) or not above the entry before it (a duplicate or a descent: each kept
  // token is attended once) is reported and not copied.
  Cursor sc = ic;                          // stage 1: the unit (of lanes 0-15) of the next pair
  int sp_pair = 0;                         // stage 1: the next pair
  int sp_t1 = -1, sp_b1 = 0, sp_g1 = 0;    // stage 1: checked position (-1: none)
  int sp_t2 = -1, sp_g2 = 0, sp_phys2 = 0; // stage 2: position and its block id
  int sp_row = -1;                         // pair c: this lane's pool row (-1: not copied)
  auto sp_stage1 = [&]() {                 // load and check the kept entries of pair sp_pair
    const int k = 2 * sp_pair + (lane >> 4);
    Cursor c = sc;
    if (lane >= 16 && k < nunits) advance(c, s_nb, a.B, a.Hkv);
    int t = -1, tp = -1;
    bool has = false, need_prev = false;
    if (k < nunits) {
      const int e = c.j * 16 + (lane & 15);
      if (e < s_len[c.b]) {
        const int32_t* list = a.kept + ((size_t)c.b * a.Hkv + c.g) * a.max_kept;
        t = __ldg(list + e);
        has = true;
        need_prev = e > 0;
        if (lane == 0 && need_prev) tp = __ldg(list + e - 1);
      }
    }
    // entry e - 1 of an entry e > 0 sits in the lane before (units of a segment are
    // consecutive and full but for the last), except for lane 0
    const int up = __shfl_up_sync(kFullMask, t, 1);
    if (lane != 0) tp = up;
    sp_t1 = -1;
    if (has) {
      if (t < 0 || t >= s_lo[c.b] || (need_prev && t <= tp)) note_error(PKV_DEV_BAD_KEPT_INDEX);
      else sp_t1 = t;
    }
    sp_b1 = c.b;
    sp_g1 = c.g;
    if (2 * sp_pair + 1 < nunits) advance(sc, s_nb, a.B, a.Hkv);
    if (2 * sp_pair + 2 < nunits) advance(sc, s_nb, a.B, a.Hkv);
    ++sp_pair;
  };
  auto sp_stage2 = [&]() {                 // stage 1 -> stage 2: the entry's block id
    sp_t2 = sp_t1;
    sp_g2 = sp_g1;
    if (sp_t1 >= 0) sp_phys2 = __ldg(a.block_tables + (size_t)sp_b1 * a.MB + (sp_t1 >> 4));
  };
  auto sp_stage3 = [&]() {                 // stage 2 -> the pool row
    sp_row = -1;
    if (sp_t2 >= 0) {
      if (sp_phys2 < 0 || sp_phys2 >= a.NB) note_error(PKV_DEV_BAD_BLOCK_ID);
      else sp_row = (sp_phys2 * a.Hkv + sp_g2) * 16 + (sp_t2 & 15);  // host checks < 2^31
    }
  };
  if constexpr (SPARSE) {
    sp_stage1();
    sp_stage2();
    sp_stage1();
  }

  // Issue unit k (the one `ic` names) into slot k % R.  Dense: lane 0 copies the K and V
  // tiles as TMA boxes.  Sparse: every lane copies chunks of the unit's kept rows.
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
          if constexpr (Q8) {
            // the K tile and both tiles' 16 row scales (64 bytes each, 64-byte aligned rows of
            // the scale pools) complete on the K barrier: the softmax needs the V scales too
            auto& Ws = warps_scales[warp];
            mbar_arrive_expect_tx(&Wb.bar_k[slot], GE::kTile + 2 * 64);
            tma_load_2d(Wt.k[slot], &a.tmap_k, 0, y, &Wb.bar_k[slot], pol);
            bulk_g2s(Ws.k[slot], a.k_scale + y, 64, &Wb.bar_k[slot], pol);
            bulk_g2s(Ws.v[slot], a.v_scale + y, 64, &Wb.bar_k[slot], pol);
            mbar_arrive_expect_tx(&Wb.bar_v[slot], GE::kTile);
            tma_load_2d(Wt.v[slot], &a.tmap_v, 0, y, &Wb.bar_v[slot], pol);
          } else {
            mbar_arrive_expect_tx(&Wb.bar_k[slot], GE::kTile);
#pragma unroll
            for (int bx = 0; bx < GE::kBoxes; ++bx)
              tma_load_2d(Wt.k[slot] + bx * 2048, &a.tmap_k, bx * 64, y, &Wb.bar_k[slot], pol);
            mbar_arrive_expect_tx(&Wb.bar_v[slot], GE::kTile);
#pragma unroll
            for (int bx = 0; bx < GE::kBoxes; ++bx)
              tma_load_2d(Wt.v[slot] + bx * 2048, &a.tmap_v, bx * 64, y, &Wb.bar_v[slot], pol);
          }
        } else {
          note_error(PKV_DEV_BAD_BLOCK_ID);
          Wb.meta[slot] = 0u;
          mbar_arrive_expect_tx(&Wb.bar_k[slot], 0);
          mbar_arrive_expect_tx(&Wb.bar_v[slot], 0);
        }
      }
      advance(ic, s_nb, a.B, a.Hkv);
    } else {
      const int r = lane & 15;
      const bool is_v = lane >= 16;
      if ((k & 1) == 0) {  // a new pair: advance the row pipeline
        sp_stage3();
        sp_stage2();
        sp_stage1();
      }
      const int pb = (k & 1) << 4;  // lanes of sp_row holding this unit's rows
      const int row = __shfl_sync(kFullMask, sp_row, pb | r);
      const bool ok = row >= 0;
      const uint32_t vmask = __ballot_sync(kFullMask, ok) & 0xffffu;  // K and V lanes agree
      // The rows arrive as 16-byte cp.async chunks into the dense tiles' swizzled layout: lane l
      // copies chunk l % CPR of rows l / CPR + RPI i.  These are ordinary per-lane instructions
      // (a bulk copy per lane with its own address costs the warp one issue per lane: ~300
      // instructions per unit, measured).  Each lane then registers its copies with the slot's
      // barriers -- the K chunks and, over INT8 pools, both rows' scales (the softmax reads the V
      // scales before the V rows land) with the K barrier, the V chunks with the V barrier --
      // before lane 0's own arrivals.
      constexpr int CPR = GE::kRow / 16;  // 16-byte chunks per row
      constexpr int RPI = 32 / CPR;       // rows one warp instruction covers
      const int cc = lane % CPR, r0 = lane / CPR;
      int rows[16 / RPI];
#pragma unroll
      for (int i = 0; i < 16 / RPI; ++i) rows[i] = __shfl_sync(kFullMask, sp_row, pb | (r0 + RPI * i));
      if constexpr (Q8) {
        auto& Ws = warps_scales[warp];
        if (ok) cp_async_4(is_v ? &Ws.v[slot][r] : &Ws.k[slot][r], (is_v ? a.v_scale : a.k_scale) + row);
      }
      const unsigned char* kb = reinterpret_cast<const unsigned char*>(a.k_cache) + cc * 16;
      const unsigned char* vb = reinterpret_cast<const unsigned char*>(a.v_cache) + cc * 16;
#pragma unroll
      for (int i = 0; i < 16 / RPI; ++i)
        if (rows[i] >= 0)
          cp_async_16(Wt.k[slot] + chunk_offset<D, SPARSE, Q8>(r0 + RPI * i, cc), kb + (size_t)rows[i] * GE::kRow, pol);
      cp_async_mbar_arrive(&Wb.bar_k[slot]);
#pragma unroll
      for (int i = 0; i < 16 / RPI; ++i)
        if (rows[i] >= 0)
          cp_async_16(Wt.v[slot] + chunk_offset<D, SPARSE, Q8>(r0 + RPI * i, cc), vb + (size_t)rows[i] * GE::kRow, pol);
      cp_async_mbar_arrive(&Wb.bar_v[slot]);
      __syncwarp();
      if (lane == 0) {
        Wb.meta[slot] = vmask;
        mbar_arrive_expect_tx(&Wb.bar_k[slot], 0);
        mbar_arrive_expect_tx(&Wb.bar_v[slot], 0);
      }
      __syncwarp();
      advance(ic, s_nb, a.B, a.Hkv);
    }
  };

  int issued = 0;
  for (; issued < nunits && issued < R; ++issued) issue(issued);
  if (!waited) {  // early prologue: the first tiles are on their way; q comes after the wait
    finish_wait();
    load_q(cc.b, cc.g);
  }
  // ask for the next range while this one's last units are still in flight
  bool requested = false;
  if (issued == nunits) {
    if (lane == 0 && tickets > 0) t_req = atomicAdd(a.ctrl, 1u);
    requested = true;
  }

  // ---- consumer state: this lane's heads are h0 = 2tq and h1 = 2tq + 1 ------------------
  uint32_t qb[2 * KS];   // q^T B fragments of the current segment
  float o[KS][4];        // O^T accumulator fragments: [m-tile][d row gq / gq+8, head h0 / h1]
  float mr0 = -INFINITY, mr1 = -INFINITY;  // running max (reference) of heads h0, h1
  float l0 = 0.f, l1 = 0.f;                // this lane's share of the running sums
  int seg_b = -1, seg_g = -1;
  int seg_slot = -1;  // partial slot of the current segment, -1: written out directly
  float* seg_logits = nullptr;  // scores mode: logit row of this lane's head h0 in the segment
  const float sl2 = a.scale_log2;
  // INT8 pools: q of the segment is prescaled by a power of two into fp16 range, so logits
  // use sl2q = sl2 over that power; o is kept in units of a V-scale reference vref that moves
  // (and rescales o) only when a unit's largest V scale exceeds it by kVrefSlack.
  float sl2q = sl2, vref = 0.f, inv_vref = 0.f;
  // INT8 pools: K codes enter q.K as the fp16 numbers 1152 + code (no subtraction per element);
  // each unit's S accumulator starts at -1152 sum_k q'_k of its head instead of 0, computed once
  // per segment by the tensor core from the same q fragments (accumulator layout: rows gq, gq + 8,
  // heads 2tq, 2tq + 1).
  float kbias[4] = {0.f, 0.f, 0.f, 0.f};
  // Dense append mode: this step's K (lanes 0-15) or V (lanes 16-31) row chunk of the current
  // segment, to be written at token L_b - 1 (pool and tile) when its unit is consumed.
  // INT8 pools: the half-warp quantizes its row when the segment begins (the INT8 append's row
  // rule: scale max|x| / 127, codes round-half-even of x / scale, both in IEEE fp32) and the
  // step writes codes and scale to the pool, the tile and the tile's scales; a row with a
  // non-finite value is reported and neither row is written.
  const bool appending = !SPARSE && a.k_new != nullptr;
  uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
  const int new_chunk = lane & 15;
  const bool new_lane = new_chunk < D / 8;
  uint2 new_codes = make_uint2(0u, 0u);  // INT8: this lane's 8 codes of the row
  float new_scale = 0.f;                 // INT8: the row's scale (K: lanes 0-15, V: 16-31)
  bool new_ok = true;                    // INT8: both rows finite

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
      if (seg_slot < 0) {
        if constexpr (SCORES) {  // the row's log-sum-exp: m is the reference l is relative to
          if (gq == 0) a.lse[row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if constexpr (Q8) {  // accumulator rows gq, gq + 8 are columns 2gq, 2gq + 1 of each 16
          const float f = inv * vref;
          __nv_bfloat16* dst = a.out + row * D + 2 * gq;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
            *reinterpret_cast<uint32_t*>(dst + mt * 16) = pack_bf16x2(o[mt][hh] * f, o[mt][2 + hh] * f);
        } else {
          __nv_bfloat16* dst = a.out + row * D + gq;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            dst[mt * 16] = __float2bfloat16_rn(o[mt][hh] * inv);
            dst[mt * 16 + 8] = __float2bfloat16_rn(o[mt][2 + hh] * inv);
          }
        }
      } else {
        const size_t e = (size_t)seg_slot * G + head;  // a flush writes G adjacent entries
        if constexpr (Q8) {
          float* dst = a.part_o + e * D + 2 * gq;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
            *reinterpret_cast<float2*>(dst + mt * 16) = make_float2(o[mt][hh] * vref, o[mt][2 + hh] * vref);
        } else {
          float* dst = a.part_o + e * D + gq;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            dst[mt * 16] = o[mt][hh];
            dst[mt * 16 + 8] = o[mt][2 + hh];
          }
        }
        if (gq == 0) a.part_ml[e] = make_float2(m, l);
      }
    }
  };

  auto begin_segment = [&](const Cursor& c) {
    seg_b = c.b;
    seg_g = c.g;
    const int nb = s_nb[c.b];
    const int seg_begin = s_start[c.b] + c.g * nb;
    // a segment inside this range is written out directly; otherwise the range's share is a
    // partial in slot 2 ridx (the segment holds the range's start) or 2 ridx + 1 (its end)
    seg_slot = (seg_begin >= u0 && seg_begin + nb <= u0 + nunits) ? -1 : 2 * ridx + (u0 >= seg_begin ? 0 : 1);
    if constexpr (SCORES)
      seg_logits = a.logits + ((size_t)c.b * a.Hq + (size_t)c.g * G + 2 * tq) * a.score_stride;
    if constexpr (Q8) {
      // q times 2^kq, with the segment's largest |q| brought into [2^14, 2^15): exact for
      // bf16 inputs, inside fp16 range (sign-cleared fp32 bit patterns order like the values)
      uint32_t mx = 0u;
#pragma unroll
      for (int i = 0; i < 2 * KS; ++i) mx = max(mx, max(qraw[i] & 0x7fff0000u, (qraw[i] << 16) & 0x7fff0000u));
      mx = __reduce_max_sync(kFullMask, mx);
      const int kq = mx == 0u ? 0 : max(-100, min(100, 141 - (int)(mx >> 23)));
      const float up = __int_as_float((127 + kq) << 23);
      sl2q = sl2 * __int_as_float((127 - kq) << 23);
#pragma unroll
      for (int i = 0; i < 2 * KS; ++i) qb[i] = pack_f16x2(bf16_lo_to_f32(qraw[i]) * up, bf16_hi_to_f32(qraw[i]) * up);
      {
        constexpr uint32_t kNeg1152 = 0xe480e480u;  // fp16x2 (-1152, -1152)
        const uint32_t ab[4] = {kNeg1152, kNeg1152, kNeg1152, kNeg1152};
#pragma unroll
        for (int i = 0; i < 4; ++i) kbias[i] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) mma_f16_m16n8k16(kbias, ab, qb[2 * ks], qb[2 * ks + 1]);
      }
      vref = 0.f;
      inv_vref = 0.f;
    } else {
#pragma unroll
      for (int i = 0; i < 2 * KS; ++i) qb[i] = qraw[i];
    }
    // only the range holding the segment's last unit (position L - 1) appends
    const bool seg_appends = appending && seg_begin + nb - 1 >= u0 && seg_begin + nb - 1 < u0 + nunits;
    if (seg_appends && new_lane) {
      const __nv_bfloat16* src = (lane >= 16 ? a.v_new : a.k_new) + ((size_t)c.b * a.Hkv + c.g) * D + new_chunk * 8;
      new_row = __ldg(reinterpret_cast<const uint4*>(src));
    }
    if constexpr (Q8) {
      if (seg_appends) {
        const uint32_t w[4] = {new_row.x, new_row.y, new_row.z, new_row.w};
        float x[8], amax = 0.f;
        bool finite = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[2 * i] = __uint_as_float(w[i] << 16);
          x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          finite &= isfinite(x[i]);
          amax = fmaxf(amax, fabsf(x[i]));
        }
#pragma unroll
        for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));  // the half
        new_ok = __all_sync(kFullMask, finite);
        if (!new_ok && lane == 0) record_error(a.err, PKV_DEV_BAD_VALUE);
        new_scale = __fdiv_rn(amax, 127.0f);
        uint32_t pk[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          int cd = 0;
          if (new_scale != 0.f) cd = max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], new_scale))));
          pk[i / 4] |= (uint32_t)(cd + 128) << (8 * (i % 4));  // stored as code + 128
        }
        new_codes = make_uint2(pk[0], pk[1]);
      }
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
      if (appending && new_ok && mask != 0u && s_len[cc.b] - 1 - tok0 < 16) {
        t_new = s_len[cc.b] - 1 - tok0;
        const size_t prow = ((size_t)Wb.phys[slot] * a.Hkv + cc.g) * 16 + t_new;  // pool row
        // the tile was read before the append: put the new K row in it and in the pool
        if constexpr (Q8) {
          // codes of elements [8c, 8c + 8) are the half (c & 1) of 16-byte chunk c / 2; both
          // rows' scales go in now (the softmax reads the V scales before the V tile lands)
          if (lane < 16 && new_lane) {
            *reinterpret_cast<uint2*>(Wt.k[slot] + chunk_offset<D, SPARSE, Q8>(t_new, new_chunk >> 1) +
                                      (new_chunk & 1) * 8) = new_codes;
            *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(a.k_pool_out) + prow * D + new_chunk * 8) =
                new_codes;
          }
          if (lane == 0) {
            warps_scales[warp].k[slot][t_new] = new_scale;
            a.k_scale_out[prow] = new_scale;
          } else if (lane == 16) {
            warps_scales[warp].v[slot][t_new] = new_scale;
            a.v_scale_out[prow] = new_scale;
          }
        } else {
          if (lane < 16 && new_lane) {
            *reinterpret_cast<uint4*>(Wt.k[slot] + chunk_offset<D, SPARSE>(t_new, new_chunk)) = new_row;
            *reinterpret_cast<uint4*>(a.k_pool_out + prow * D + new_chunk * 8) = new_row;
          }
        }
        __syncwarp();
      }
    }
    if (mask != 0u) {
      // -- S^T = K q^T: 16 tokens x 8 heads --------------------------------------------------
      float c[4] = {kbias[0], kbias[1], kbias[2], kbias[3]};  // zero but for INT8 pools
      const uint32_t kbase = smem_u32(Wt.k[slot]);
      float fk0 = sl2, fk1 = sl2;  // logit factor of tokens gq and gq + 8
      if constexpr (Q8) {
        // int8 rows: one ldmatrix yields two k-steps; each lane holds 4 consecutive columns
        // of a row per matrix, the order q was loaded in; the codes enter as 1152 + code
#pragma unroll
        for (int pp = 0; pp < KS / 2; ++pp) {
          uint32_t r[4];
          ldsm_x4(kbase + chunk_offset<D, SPARSE, Q8>(k_row, 2 * pp + k_half), r);
          const uint32_t f0 = r[0], f1 = r[1], f2 = r[2], f3 = r[3];  // bytes code + 128
          const uint32_t a0[4] = {i8x2_to_biased_f16x2<0x4140>(f0), i8x2_to_biased_f16x2<0x4140>(f1),
                                  i8x2_to_biased_f16x2<0x4342>(f0), i8x2_to_biased_f16x2<0x4342>(f1)};
          mma_f16_m16n8k16(c, a0, qb[4 * pp], qb[4 * pp + 1]);
          const uint32_t a1[4] = {i8x2_to_biased_f16x2<0x4140>(f2), i8x2_to_biased_f16x2<0x4140>(f3),
                                  i8x2_to_biased_f16x2<0x4342>(f2), i8x2_to_biased_f16x2<0x4342>(f3)};
          mma_f16_m16n8k16(c, a1, qb[4 * pp + 2], qb[4 * pp + 3]);
        }
        fk0 = warps_scales[warp].k[slot][gq] * sl2q;
        fk1 = warps_scales[warp].k[slot][gq + 8] * sl2q;
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t af[4];
          ldsm_x4(kbase + chunk_offset<D, SPARSE>(k_row, 2 * ks + k_half), af);
          mma_bf16_m16n8k16(c, af, qb[2 * ks], qb[2 * ks + 1]);
        }
      }
      // c[0] = (token gq, head h0), c[1] = (gq, h1), c[2] = (gq + 8, h0), c[3] = (gq + 8, h1)
      const bool t0 = (mask >> gq) & 1u;
      const bool t1 = (mask >> (gq + 8)) & 1u;
      const bool v0 = 2 * tq < G, v1 = 2 * tq + 1 < G;
      const float s00 = (t0 && v0) ? c[0] * fk0 : -INFINITY;
      const float s01 = (t0 && v1) ? c[1] * fk0 : -INFINITY;
      const float s10 = (t1 && v0) ? c[2] * fk1 : -INFINITY;
      const float s11 = (t1 && v1) ? c[3] * fk1 : -INFINITY;
      if constexpr (SCORES) {  // keep the attended keys' logits for the score step
        const int tok = (s_first[cc.b] + cc.j) * 16 + gq;
        float* lg = seg_logits + tok;
        if (tok < a.score_stride) {
          if (t0 && v0) lg[0] = s00;
          if (t0 && v1) lg[a.score_stride] = s01;
        }
        if (tok + 8 < a.score_stride) {
          if (t1 && v0) lg[8] = s10;
          if (t1 && v1) lg[a.score_stride + 8] = s11;
        }
      }
      // lazy running max: move it only when this unit's max is well above it.  Each lane checks
      // its own two tokens first; the unit's maxima (shuffles over the 8 token rows) are needed
      // only when some lane's logit, or (INT8 pools) V scale, is past its reference.
      float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
      // INT8 pools: the V scales of the attended tokens, and their largest
      float vs0 = 0.f, vs1 = 0.f;
      float vm = 0.f;
      if constexpr (Q8) {
        vs0 = t0 ? warps_scales[warp].v[slot][gq] : 0.f;
        vs1 = t1 ? warps_scales[warp].v[slot][gq + 8] : 0.f;
        vm = fmaxf(vs0, vs1);
      }
      bool g0 = mx0 > mr0 + kRescaleSlack, g1 = mx1 > mr1 + kRescaleSlack;
      bool gv = Q8 && vm > vref * kVrefSlack;
      if (__any_sync(kFullMask, g0 || g1 || gv)) {
#pragma unroll
        for (int m = 4; m <= 16; m <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, m));
          mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, m));
        }
        g0 = mx0 > mr0 + kRescaleSlack;
        g1 = mx1 > mr1 + kRescaleSlack;
        if constexpr (Q8) {  // warp-uniform: the scales of a token are the same in its 4 lanes
#pragma unroll
          for (int m = 4; m <= 16; m <<= 1) vm = fmaxf(vm, __shfl_xor_sync(kFullMask, vm, m));
          gv = vm > vref * kVrefSlack;
        }
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
        if constexpr (Q8) {
          if (gv) {  // o moves to the new V reference (o is zero while vref is)
            const float fv = vref > 0.f ? vref / vm : 0.f;
            al0 *= fv;
            al1 *= fv;
            vref = vm;
            inv_vref = 1.f / vm;
          }
        }
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
      // -- P^T as B fragments (tokens x heads -> heads x tokens) ---------------------------
      // INT8 pools: P times each token's V scale over vref (at most 2^8 * slack) as one fp16
      // term (11 significant bits, below the bf16 output's rounding);
      // bf16: a hi + lo pair of bf16 terms (8 bits alone would not be)
      uint32_t hA, hB, lA = 0u, lB = 0u;
      if constexpr (Q8) {
        const float r0 = vs0 * inv_vref, r1 = vs1 * inv_vref;
        hA = pack_f16x2(p00 * r0, p01 * r0);
        hB = pack_f16x2(p10 * r1, p11 * r1);
      } else {
        hA = pack_bf16x2(p00, p01);  // token gq
        hB = pack_bf16x2(p10, p11);  // token gq + 8
        lA = pack_bf16x2(p00 - bf16_lo_to_f32(hA), p01 - bf16_hi_to_f32(hA));
        lB = pack_bf16x2(p10 - bf16_lo_to_f32(hB), p11 - bf16_hi_to_f32(hB));
      }
      const uint32_t bh0 = movmatrix_trans(hA), bh1 = movmatrix_trans(hB);
      const uint32_t bl0 = Q8 ? 0u : movmatrix_trans(lA), bl1 = Q8 ? 0u : movmatrix_trans(lB);
      if (!__all_sync(kFullMask, mbar_wait_bounded(&Wb.bar_v[slot], parity, a.timeout_ns))) {
        if (lane == 0) record_error(a.err, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
        break;
      }
      if (t_new >= 0) {  // append mode: the new V row, into the tile and the pool
        const size_t prow = ((size_t)Wb.phys[slot] * a.Hkv + cc.g) * 16 + t_new;
        if (lane >= 16 && new_lane) {
          if constexpr (Q8) {
            *reinterpret_cast<uint2*>(Wt.v[slot] + chunk_offset<D, SPARSE, Q8>(t_new, new_chunk >> 1) +
                                      (new_chunk & 1) * 8) = new_codes;
            *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(a.v_pool_out) + prow * D + new_chunk * 8) =
                new_codes;
          } else {
            *reinterpret_cast<uint4*>(Wt.v[slot] + chunk_offset<D, SPARSE>(t_new, new_chunk)) = new_row;
            *reinterpret_cast<uint4*>(a.v_pool_out + prow * D + new_chunk * 8) = new_row;
          }
        }
        __syncwarp();
      }
      if constexpr (!Q8) {
        if (mask != 0xffffu) {
          // rows of tokens outside the attended set may hold anything (even NaN): zero them,
          // since the tensor core would turn 0 * NaN into NaN (int8 codes are always finite)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int t = 2 * i + (lane >> 4);
            const int c = lane & 15;  // chunk (16 bytes) of the row
            if (!((mask >> t) & 1u) && c < D / 8)
              *reinterpret_cast<uint4*>(Wt.v[slot] + chunk_offset<D, SPARSE>(t, c)) = make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
      }
      // -- O^T += V^T P^T -------------------------------------------------------------------
      const uint32_t vbase = smem_u32(Wt.v[slot]);
      if constexpr (Q8) {
        // transposed int8 ldmatrix: each lane gets columns 2gq, 2gq + 1 of tokens 2tq, 2tq + 1;
        // columns 2gq and 2gq + 1 become accumulator rows gq and gq + 8 of the 16-column tile
#pragma unroll
        for (int pp = 0; pp < KS / 2; ++pp) {
          uint32_t r[4];
          ldsm_x4_trans(vbase + chunk_offset<D, SPARSE, Q8>(k_row, 2 * pp + k_half), r);
          const uint32_t f0 = r[0], f1 = r[1], f2 = r[2], f3 = r[3];  // bytes code + 128
          const uint32_t a0[4] = {i8x2_to_f16x2<0x4240>(f0), i8x2_to_f16x2<0x4341>(f0),
                                  i8x2_to_f16x2<0x4240>(f1), i8x2_to_f16x2<0x4341>(f1)};
          mma_f16_m16n8k16(o[2 * pp], a0, bh0, bh1);
          const uint32_t a1[4] = {i8x2_to_f16x2<0x4240>(f2), i8x2_to_f16x2<0x4341>(f2),
                                  i8x2_to_f16x2<0x4240>(f3), i8x2_to_f16x2<0x4341>(f3)};
          mma_f16_m16n8k16(o[2 * pp + 1], a1, bh0, bh1);
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t av[4];
          ldsm_x4_trans(vbase + chunk_offset<D, SPARSE>(v_row, 2 * mt + v_half), av);
          mma_bf16_m16n8k16(o[mt], av, bh0, bh1);
          mma_bf16_m16n8k16(o[mt], av, bl0, bl1);
        }
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
    } else if (!requested) {
      if (lane == 0 && tickets > 0) t_req = atomicAdd(a.ctrl, 1u);
      requested = true;
    }
    advance(cc, s_nb, a.B, a.Hkv);
  }

  if (aborted) {  // let the copies in flight land before the CTA's shared memory goes away
    if constexpr (SPARSE) cp_async_wait_all();
    for (int kk = k; kk < issued; ++kk) {
      (void)mbar_wait_bounded(&Wb.bar_k[kk % R], (uint32_t)(kk / R) & 1u, a.timeout_ns);
      (void)mbar_wait_bounded(&Wb.bar_v[kk % R], (uint32_t)(kk / R) & 1u, a.timeout_ns);
    }
  } else {
    flush();
    rid = take_ticket();
  }
  }  // ranges
  finish_wait();  // a warp with no range still ends after the previous kernel
  if (lane == 0 && n_taken != 0u) atomicAdd(a.ctrl + 1, n_taken);
}

// Log-sum-exp merge of the partials of every (sequence, query head) row that more than one
// range touched.  A CTA of W warps serves W / wpr rows with wpr = 2^wpr_log2 warps each:
// warp `sub` of a row combines its partials sub, sub + wpr, sub + 2 wpr, ... and the row's
// first warp combines the wpr results through shared memory.  Also writes the zero row of
// empty sequences, checks that every tail chunk was taken exactly once and re-arms the
// ticket counters for the next call.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
decode_merge_kernel(const DecodeArgs a, int group, int wpr_log2) {
  constexpr int EPW = D / 32;
  constexpr int W = kMergeWarps;
  __shared__ float s_acc[W][D];
  __shared__ float2 s_ml[W];
  // With a.merge_trigger_early the next kernel on the stream may launch at once: every kernel
  // of this library waits for this one (griddepcontrol.wait) before it reads what this one
  // writes, and an early decode prologue reads only inputs its caller has declared final.  The
  // next decode's CTAs then take the SM slots the split kernel's last warps free and start
  // their tile copies there, instead of starting after this kernel's wait.
  if (a.merge_trigger_early) grid_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wpr = 1 << wpr_log2;
  const int sub = warp & (wpr - 1);
  const int row = blockIdx.x * (W >> wpr_log2) + (warp >> wpr_log2);
  // What this row needs (uniform over its warps; no early exit before the block barrier):
  // nothing (written by the split kernel, or past the last row), a zero row, or a merge of
  // np partials.  The partition follows from the lengths (inputs the split kernel does not
  // write, final before it started), so small batches work it out, and prefetch their first
  // partials into L2, before the split kernel ends.
  const bool sparse = a.max_kept > 0;
  const int rrow = min(row, a.B * a.Hq - 1);
  const int b = rrow / a.Hq;
  const int g = (rrow - b * a.Hq) / group;
  const int head = row - (row / group) * group;
  int32_t part[kPartFields];
  int np = 0, r0 = 0, slot0 = 0;
  bool zero_row = false;
  auto describe = [&](int before, int total, int nb) {
    make_partition(part, total * a.Hkv, a.workers, a);
    if (row >= a.B * a.Hq) return;
    if (nb == 0) {
      zero_row = true;
      return;
    }
    const int seg = before * a.Hkv + g * nb;
    const int rid0 = range_of(part, seg);
    r0 = range_index(part, rid0);
    np = range_index(part, range_of(part, seg + nb - 1)) - r0 + 1;
    if (np == 1) np = 0;
    // partial i of the row: range r0 + i (in unit order), slot 2 (r0 + i), except that the
    // segment is the second one range r0 touches (slot 2 r0 + 1) when it starts inside it
    slot0 = 2 * r0 + (range_start(part, rid0) < seg ? 1 : 0);
  };
  auto entry = [&](int i) -> size_t {
    return (size_t)(i == 0 ? slot0 : 2 * (r0 + i)) * group + head;
  };
  if (a.B <= kMergeScanMaxBatch) {
    int before = 0, total = 0, nb = 0;  // units of the sequences before b, of all, of b
    for (int base = 0; base < a.B; base += 32) {
      const int bb = base + lane;
      int v = 0;
      if (bb < a.B) v = sparse ? seq_units<true>(a, bb).nb : seq_units<false>(a, bb).nb;
      const int own = __shfl_sync(kFullMask, v, (b - base) & 31);
      if (b >= base && b < base + 32) nb = own;
      int sa = v, sb = bb < b ? v : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sa += __shfl_xor_sync(kFullMask, sa, o);
        sb += __shfl_xor_sync(kFullMask, sb, o);
      }
      total += sa;
      before += sb;
    }
    describe(before, total, nb);
    // this warp's first batch of partials (see below): lane 8j + i, i < 4, prefetches a
    // quarter of partial j's o row (512 bytes at d = 128), lane 8j + 4 its (m, l)
    const int j = lane >> 3, q = lane & 7;
    for (int jj = j; jj < 8; jj += 4) {
      const int i = sub + wpr * jj;
      if (i < np) {
        const size_t en = entry(i);
        if (q < 4) prefetch_l2(a.part_o + en * D + q * (D / 4));
        else if (q == 4) prefetch_l2(a.part_ml + en);
      }
    }
  }
  grid_dependency_wait();  // the split kernel's partials (and, for large batches, its record)
  if (!a.merge_trigger_early) grid_launch_dependents();
  if (a.B > kMergeScanMaxBatch) {
    // the record holds unit starts (already times Hkv) and unit counts per sequence
    const int last = a.B - 1;
    describe(__ldcg(a.layout + b) / a.Hkv,
             (__ldcg(a.layout + last) + a.Hkv * __ldcg(a.layout + a.B + last)) / a.Hkv,
             __ldcg(a.layout + a.B + b));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (a.ctrl[1] != (uint32_t)part[kPartTickets]) record_error(a.err, PKV_DEV_DIRTY_WORKSPACE);
    a.ctrl[0] = 0u;
    a.ctrl[1] = 0u;
  }
  // this warp's partials i = sub + wpr p, p < npw, in batches of 8.  Every lane loads the
  // batch's (m, l) pairs (one broadcast transaction each) together with its slice of the
  // batch's o rows, so a batch costs one memory round trip.
  const int npw = np > sub ? (np - sub + wpr - 1) / wpr : 0;
  float M = -INFINITY, L = 0.f;
  float acc[EPW];
#pragma unroll
  for (int e = 0; e < EPW; ++e) acc[e] = 0.f;
  for (int pb = 0; pb < npw; pb += 8) {
    float2 ml[8];
    float x[8][EPW];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ml[j] = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int e = 0; e < EPW; ++e) x[j][e] = 0.f;
      if (pb + j < npw) {
        const size_t en = entry(sub + wpr * (pb + j));
        ml[j] = __ldcg(a.part_ml + en);
        const float* src = a.part_o + en * D + lane * EPW;
        if constexpr (EPW == 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
          x[j][0] = v.x; x[j][1] = v.y; x[j][2] = v.z; x[j][3] = v.w;
        } else {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
          x[j][0] = v.x; x[j][1] = v.y;
        }
      }
    }
    float gmax = M;
#pragma unroll
    for (int j = 0; j < 8; ++j) gmax = fmaxf(gmax, ml[j].x);
    const float mref = (gmax == -INFINITY) ? 0.f : gmax;
    const float carry = exp2f(M - mref);  // rescale what earlier batches accumulated
    L *= carry;
#pragma unroll
    for (int e = 0; e < EPW; ++e) acc[e] *= carry;
    M = gmax;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float w = exp2f(ml[j].x - mref);  // 0 for the padding entries
      L += w * ml[j].y;
#pragma unroll
      for (int e = 0; e < EPW; ++e) acc[e] += w * x[j][e];
    }
  }
  float m_ref = (M == -INFINITY) ? 0.f : M;  // the reference L is relative to
  if (wpr > 1) {  // (uniform over the CTA) combine the row's wpr results
    if (lane == 0) s_ml[warp] = make_float2(M, L);
#pragma unroll
    for (int e = 0; e < EPW; ++e) s_acc[warp][lane * EPW + e] = acc[e];
    __syncthreads();
    if (sub != 0) return;
    float Mg = -INFINITY;
    for (int w = 0; w < wpr; ++w) Mg = fmaxf(Mg, s_ml[warp + w].x);
    const float mref = (Mg == -INFINITY) ? 0.f : Mg;
    m_ref = mref;
    L = 0.f;
#pragma unroll
    for (int e = 0; e < EPW; ++e) acc[e] = 0.f;
    for (int w = 0; w < wpr; ++w) {
      const float f = exp2f(s_ml[warp + w].x - mref);  // 0 for a warp without partials
      L += f * s_ml[warp + w].y;
#pragma unroll
      for (int e = 0; e < EPW; ++e) acc[e] += f * s_acc[warp + w][lane * EPW + e];
    }
  }
  if (np == 0 && !zero_row) return;
  if (a.lse != nullptr && lane == 0)  // scores mode: the row's natural log-sum-exp
    a.lse[row] = L > 0.f ? (m_ref + log2f(L)) * kLn2 : -INFINITY;
  __nv_bfloat16* dst = a.out + (size_t)row * D + lane * EPW;
  const float inv = L > 0.f ? 1.f / L : 0.f;  // a zero row has L = 0 and acc = 0
#pragma unroll
  for (int e = 0; e < EPW; e += 2) {
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

// The score step ([novita] "2. Attention modification": with each row's max and sum from the
// attention pass, every attended key's probability is exp(s - m) / l = exp(s - lse); a key's
// score adds the probabilities of the G query heads sharing its kv head):
//   scores[b, g, t] += sum_i 2^(logit[b, gG + i, t] - lse[b, gG + i] log2 e)
// over the attended t < score_stride.  A CTA covers 1024 keys of one (b, g); a thread four
// consecutive keys, as 16-byte loads and stores when the rows allow it (16-byte aligned
// buffers, score_stride % 4 == 0).
constexpr int kScoreThreads = 256;
constexpr int kScoreKeys = 4 * kScoreThreads;

__global__ void __launch_bounds__(kScoreThreads) decode_score_kernel(const DecodeArgs a, int group, int tiles) {
  const int seg = blockIdx.x / tiles;  // b * Hkv + g
  const int tile = blockIdx.x - seg * tiles;
  grid_dependency_wait();  // the logits and log-sum-exps of the decode
  grid_launch_dependents();
  const int b = seg / a.Hkv;
  const int g = seg - b * a.Hkv;
  int L = a.context_lens[b];
  if (L < 0 || L > a.MB * 16) L = 0;  // reported by the split kernel
  const int start = (a.window > 0 && L > a.window) ? L - a.window : 0;
  const int end = min(L, a.score_stride);
  const int t0 = (start & ~3) + tile * kScoreKeys + 4 * (int)threadIdx.x;  // keys t0 .. t0 + 3
  if (t0 >= end || t0 + 4 <= start) return;
  const size_t row0 = (size_t)b * a.Hq + (size_t)g * group;
  float* dst = a.scores + (size_t)seg * a.score_stride + t0;
  const bool vec = (a.score_stride & 3) == 0 && t0 >= start && t0 + 4 <= end &&
                   ((reinterpret_cast<uintptr_t>(a.scores) | reinterpret_cast<uintptr_t>(a.logits)) & 15u) == 0;
  float sum[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i = 0; i < group; ++i) {
    const float lse2 = a.lse[row0 + i] * kLog2e;
    const float* src = a.logits + (row0 + i) * a.score_stride + t0;
    if (vec) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      sum[0] += exp2f(v.x - lse2);
      sum[1] += exp2f(v.y - lse2);
      sum[2] += exp2f(v.z - lse2);
      sum[3] += exp2f(v.w - lse2);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (t0 + e >= start && t0 + e < end) sum[e] += exp2f(src[e] - lse2);
    }
  }
  if (vec) {
    float4 o = *reinterpret_cast<float4*>(dst);
    o.x += sum[0];
    o.y += sum[1];
    o.z += sum[2];
    o.w += sum[3];
    *reinterpret_cast<float4*>(dst) = o;
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (t0 + e >= start && t0 + e < end) dst[e] += sum[e];
  }
}

}  // namespace

DecodeKernel decode_kernel(int head_dim, int group, bool sparse, bool scores, bool q8) {
  const DecodeKernel none{nullptr, nullptr, nullptr, head_dim, group, sparse, scores, q8};
  if (group < 1 || group > kMaxGroup || (sparse && scores)) return none;
  const void* score = scores ? (const void*)decode_score_kernel : nullptr;
  if (head_dim == 128)
    return DecodeKernel{q8 ? (scores   ? (const void*)decode_split_kernel<128, false, true, true>
                              : sparse ? (const void*)decode_split_kernel<128, true, false, true>
                                       : (const void*)decode_split_kernel<128, false, false, true>)
                        : sparse ? (const void*)decode_split_kernel<128, true, false, false>
                        : scores ? (const void*)decode_split_kernel<128, false, true, false>
                                 : (const void*)decode_split_kernel<128, false, false, false>,
                        (const void*)decode_merge_kernel<128>, score, 128, group, sparse, scores, q8};
  if (head_dim == 64)
    return DecodeKernel{q8 ? (scores   ? (const void*)decode_split_kernel<64, false, true, true>
                              : sparse ? (const void*)decode_split_kernel<64, true, false, true>
                                       : (const void*)decode_split_kernel<64, false, false, true>)
                        : sparse ? (const void*)decode_split_kernel<64, true, false, false>
                        : scores ? (const void*)decode_split_kernel<64, false, true, false>
                                 : (const void*)decode_split_kernel<64, false, false, false>,
                        (const void*)decode_merge_kernel<64>, score, 64, group, sparse, scores, q8};
  return none;
}

size_t decode_smem_bytes(int head_dim, bool sparse, int batch) {
  (void)sparse;
  if (head_dim != 128 && head_dim != 64) return 0;
  // dynamic part only: the per-sequence arrays (the tile rings are static)
  return sizeof(int32_t) * (5 * (size_t)batch + 1);
}

cudaError_t launch_decode(const DecodeKernel& k, const DecodeArgs& a, int grid, size_t smem,
                          int merge_wpr_log2, cudaStream_t stream) {
  DecodeArgs args = a;
  args.G = k.group;
  void* split_params[] = {&args};
  cudaError_t e = launch_pdl(k.split, dim3(grid), dim3(kDecodeWarps * 32), smem, stream, split_params);
  if (e != cudaSuccess) return e;
  int group = k.group;
  int wpr_log2 = merge_wpr_log2;
  void* merge_params[] = {&args, &group, &wpr_log2};
  const long long rows = (long long)a.B * a.Hq;
  const int rows_per_cta = kMergeWarps >> merge_wpr_log2;
  const long long mgrid = (rows + rows_per_cta - 1) / rows_per_cta;
  if (mgrid == 0) return cudaSuccess;
  e = launch_pdl(k.merge, dim3((unsigned)mgrid), dim3(kMergeWarps * 32), 0, stream, merge_params);
  if (e != cudaSuccess || !k.scores) return e;
  // score step: tiles of 256 keys over the longest attended range any sequence can have
  long long span = (long long)a.MB * 16;
  if (a.window > 0 && a.window < span) span = a.window;
  if (a.score_stride < span) span = a.score_stride;
  int tiles = (int)((span + 3 + kScoreKeys - 1) / kScoreKeys);  // +3: the start rounds down to 4
  if (tiles < 1) tiles = 1;
  void* score_params[] = {&args, &group, &tiles};
  const long long sgrid = (long long)a.B * a.Hkv * tiles;
  return launch_pdl(k.score, dim3((unsigned)sgrid), dim3(kScoreThreads), 0, stream, score_params);
}

}  // namespace pkv
