// kernels.h -- argument records and launchers shared between the C-ABI layer (api.cu) and
// the kernel translation units.  Internal to the library; the public boundary is pkv.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Split-K decode.  The flattened (sequence, kv head, 16-token unit) list is cut into one
// slice of P units per worker warp.  A slice is a static head of S units, processed by the
// warp of the same index, and cpw tail chunks of halving length that warps take from a
// shared ticket counter once their head is done, so warps on faster SMs absorb the work of
// slower ones.  Heads and chunks are the "ranges" of the partition; which warp runs a range never
// changes what it computes, and its partial results go to fixed slots of the range.
struct DecodeArgs {
  CUtensorMap tmap_k;            // dense mode: the K pool as a 2-D [NB*Hkv*16, D] bf16 tensor,
  CUtensorMap tmap_v;            //   box 64 x 16, 128-byte swizzle (likewise V); INT8 pools:
                                 //   [NB*Hkv*16, D] bytes, box D x 16, swizzle of D bytes
  const __nv_bfloat16* q;        // [B, Hq, D]
  const __nv_bfloat16* k_cache;  // [NB, Hkv, 16, D]
  const __nv_bfloat16* v_cache;
  const int32_t* block_tables;   // [B, MB]
  const int32_t* context_lens;   // [B]
  const int32_t* kept;           // [B, Hkv, max_kept] (sparse mode)
  const int32_t* kept_lens;      // [B]               (sparse mode)
  const __nv_bfloat16* k_new;    // [B, Hkv, D] this step's token (dense append mode) or nullptr
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool_out;     // the pools again, writable (append mode)
  __nv_bfloat16* v_pool_out;
  __nv_bfloat16* out;            // [B, Hq, D]
  uint32_t* ctrl;                // [2]: tail-chunk ticket counter, chunks taken; zero between calls
  int32_t* layout;               // [2B]: unit start (times Hkv) and units of each sequence, for large B
  float2* part_ml;               // [2 ranges, G] (running max in log2 units, running sum)
  float* part_o;                 // [2 ranges, G, D] unnormalised partial outputs
  const float* k_scale;          // INT8 pools: [NB, Hkv, 16] fp32 scale of each K row
  const float* v_scale;          //   (likewise V); the pools then hold INT8 codes (bytes code + 128)
  float* k_scale_out;            // INT8 append mode: the scale pools again, writable
  float* v_scale_out;
  float* logits;                 // scores mode: [B, Hq, score_stride] base-2 logits of attended keys
  float* lse;                    // scores mode: [B, Hq] natural log-sum-exp of each row
  float* scores;                 // scores mode: [B, Hkv, score_stride] accumulated scores
  int score_stride;              // scores mode: row length of logits and scores
  int32_t* err;                  // device error word or nullptr
  int B, Hq, Hkv, NB, MB, max_kept, window;
  int workers;                   // worker warps of the split grid
  int min_units;                 // lower bound of the slice length P
  int min_busy_pct;              // the floor yields to keep this share of the workers busy (0: never)
  int tail_pct;                  // share of a slice given out as tail chunks, in percent
  int chunk_min;                 // lower bound of a chunk length (>= the tile ring depth)
  int cpw_cap;                   // upper bound of the chunks per slice (workspace slots)
  int G;                         // query heads per kv head (1..kMaxGroup)
  int early;                     // 1: the pools, tables, lengths and kept lists are final before the
                                 //   previous kernel on the stream ends (PKV_DECODE_INPUTS_READY): the
                                 //   split kernel partitions and starts its first tile copies before
                                 //   waiting for that kernel; q, new rows and the workspace after it
  int merge_trigger_early;       // 1: the merge kernel lets the next kernel launch at its start, not
                                 //   after its wait (set for early bf16 calls, see decode_common)
  float scale_log2;              // scale * log2(e): logits are kept in base-2 units
  unsigned long long timeout_ns; // bound of every mbarrier wait
};

// Partition record: computed from the total unit count and the worker count alone, so every
// split CTA and every merge warp derives the same one.
// kPartOff + c holds O_c, the start of tail chunk c within the tail (c = 0..cpw).
enum PartField { kPartTotal = 0, kPartP, kPartS, kPartTail, kPartCpw, kPartNfull, kPartTickets, kPartWorkers, kPartOff };
constexpr int kMaxTailChunksLimit = 7;  // cpw bound of the record (and of the range-id packing)
constexpr int kPartFields = kPartOff + kMaxTailChunksLimit + 1;

// Tuning knobs (compile-time; every setting computes the same result).
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 1
#endif
#ifndef PKV_RING_D128
#define PKV_RING_D128 2  // K/V tile pairs in flight per worker warp at head_dim 128
#endif
#ifndef PKV_RING_D64
#define PKV_RING_D64 4
#endif

#ifndef PKV_RING_Q8_D128
#define PKV_RING_Q8_D128 2  // INT8 K/V tile pairs in flight per worker warp at head_dim 128
#endif
#ifndef PKV_RING_Q8_D64
#define PKV_RING_Q8_D64 4
#endif

#ifndef PKV_RING_SPARSE_D128
#define PKV_RING_SPARSE_D128 2  // gather form of the sparse decode (bf16 and INT8) at head_dim 128
#endif

#ifndef PKV_Q8_MIN_CTAS
#define PKV_Q8_MIN_CTAS 12  // INT8 decode: resident CTAs per SM the register budget must allow (0: no bound)
#endif

#ifndef PKV_MIN_UNITS
#define PKV_MIN_UNITS 16  // lower bound of a worker slice, in 16-token units
#endif
#ifndef PKV_MIN_BUSY_PCT
#define PKV_MIN_BUSY_PCT 70  // the slice floor yields to keep this share of the workers busy (0: never)
#endif
// The dense decode over INT8 pools spends more instructions per unit: there every worker takes
// a slice (measured: the 28-layer qwen step over INT8 pools 0.913 -> 0.835 ms, the sparse step
// over INT8 pools 1.098 -> 1.040 ms), while the bf16 decode keeps the floor (all workers busy
// made the qwen step 0.911 -> 0.973 ms).  The score-emitting decode keeps the plain decode's
// partition, so its output stays bit-identical to the plain call's.
#ifndef PKV_MIN_UNITS_Q8
#define PKV_MIN_UNITS_Q8 16
#endif
#ifndef PKV_MIN_BUSY_PCT_Q8
#define PKV_MIN_BUSY_PCT_Q8 100
#endif
// A 10 % tail (none for the llama8b-shaped layer's 35-unit slices, one chunk from 60 units up):
// the INT8 layer 64.3 -> 60.9 us, with scores 74.1 -> 69.8 us (20 % gave those slices one
// 7-unit chunk each).
#ifndef PKV_TAIL_PCT_Q8
#define PKV_TAIL_PCT_Q8 10
#endif
#ifndef PKV_CHUNK_MIN_Q8
#define PKV_CHUNK_MIN_Q8 6
#endif
#ifndef PKV_MIN_UNITS_SPARSE
#define PKV_MIN_UNITS_SPARSE 8  // the same for the gather form of the sparse decode (measured)
#endif
#ifndef PKV_TAIL_PCT
#define PKV_TAIL_PCT 20   // share of a slice handed out dynamically
#endif
#ifndef PKV_MIN_BUSY_PCT_SPARSE
#define PKV_MIN_BUSY_PCT_SPARSE 70  // the busy share of the gather form
#endif
// over INT8 pools every worker takes a slice (one sparse layer: 28.9 -> 27.8 us; bf16 unchanged)
#ifndef PKV_MIN_BUSY_PCT_SPARSE_Q8
#define PKV_MIN_BUSY_PCT_SPARSE_Q8 100
#endif
#ifndef PKV_TAIL_PCT_SPARSE
#define PKV_TAIL_PCT_SPARSE 30  // the same for the gather form of the sparse decode (measured)
#endif
#ifndef PKV_CHUNK_MIN
#define PKV_CHUNK_MIN 6   // shortest tail chunk, in units (at least the tile ring depth)
#endif
#ifndef PKV_MAX_TAIL_CHUNKS
#define PKV_MAX_TAIL_CHUNKS 4
#endif
#ifndef PKV_MERGE_PARTIALS_PER_WARP
#define PKV_MERGE_PARTIALS_PER_WARP 16 // merge warps per row grow while a warp would take more
#endif
// INT8 decodes, where every worker takes a slice and rows have more partials: more merge warps
// per row (measured against 16: qwen INT8 step 0.833 -> 0.784 ms, sparse INT8 step 1.035 ->
// 1.008 ms; for bf16 the qwen step lost 1 % at 4 and 6 % at 8, so it keeps 16).
#ifndef PKV_MERGE_PARTIALS_PER_WARP_Q8
#define PKV_MERGE_PARTIALS_PER_WARP_Q8 4
#endif

constexpr int kDecodeWarps = PKV_DECODE_WARPS;  // worker warps per CTA
constexpr int kMaxWorkers = 2048;    // worker warps of a decode grid at most (sizes the workspace)
constexpr int kMergeWarps = 8;
constexpr int kMaxGroup = 8;         // query heads per kv head handled by one fragment

// Kernel handles of one (head_dim, group, sparse, scores, INT8) instantiation.
struct DecodeKernel {
  const void* split;
  const void* merge;
  const void* score;  // scores mode: adds the step's probabilities into the scores
  int head_dim, group;
  bool sparse, scores, q8;
};

// Returns a struct with split == nullptr when the combination is unsupported (scores mode
// and INT8 pools exist for dense decode only, and not together).
DecodeKernel decode_kernel(int head_dim, int group, bool sparse, bool scores = false, bool q8 = false);
size_t decode_smem_bytes(int head_dim, bool sparse, int batch);
// merge_wpr_log2: log2 of the merge warps per output row (0..3).
cudaError_t launch_decode(const DecodeKernel& k, const DecodeArgs& a, int grid, size_t smem,
                          int merge_wpr_log2, cudaStream_t stream);

// kv append / compaction / top-k selection.  kvops_device_setup() sets the kernels'
// attributes on the current device (called once per device by the C ABI).
cudaError_t kvops_device_setup();
cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                             const int64_t* slots, int64_t T, int Hkv, int D, int NB,
                             int32_t* err, cudaStream_t stream);
cudaError_t launch_kv_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                                const void* k, const void* v, const int64_t* slots, int64_t T, int Hkv,
                                int D, int NB, int32_t* err, cudaStream_t stream);
cudaError_t launch_kv_compact(void* dk, void* dv, const int32_t* dbt, int dNB, int dMB,
                              const void* sk, const void* sv, const int32_t* sbt,
                              const int32_t* lens, const int32_t* kept, const int32_t* kept_lens,
                              int max_kept, int B, int Hkv, int D, int sNB, int sMB, int early,
                              int32_t* err, cudaStream_t stream);
cudaError_t launch_kv_rolling_admit(void* k_cache, void* v_cache, const int32_t* bt, int NB, int MB,
                                    int32_t* slot_pos, float* slot_score, int32_t* kept_lens,
                                    const int32_t* lens, const void* k_new, const void* v_new, int B,
                                    int Hkv, int D, int capacity, int n_sink, int n_recent, int early,
                                    int32_t* err, cudaStream_t stream);
// INT8 pools: codes [NB, Hkv, 16, D] (bytes code + 128) with row scales [NB, Hkv, 16] fp32 moving with them.
cudaError_t launch_kv_compact_q8(void* dk, void* dv, float* dks, float* dvs, const int32_t* dbt, int dNB,
                                 int dMB, const void* sk, const void* sv, const float* sks, const float* svs,
                                 const int32_t* sbt, const int32_t* lens, const int32_t* kept,
                                 const int32_t* kept_lens, int max_kept, int B, int Hkv, int D, int sNB,
                                 int sMB, int early, int32_t* err, cudaStream_t stream);
cudaError_t launch_kv_rolling_admit_q8(void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                       const int32_t* bt, int NB, int MB, int32_t* slot_pos, float* slot_score,
                                       int32_t* kept_lens, const int32_t* lens, const void* k_new,
                                       const void* v_new, int B, int Hkv, int D, int capacity, int n_sink,
                                       int n_recent, int early, int32_t* err, cudaStream_t stream);
cudaError_t launch_select_topk(int32_t* kept_out, int32_t* kept_lens_out, const float* scores,
                               int stride, const int32_t* lens, int B, int Hkv, int n_sink,
                               int n_recent, int k_top, int early, int32_t* err, cudaStream_t stream);

// Prefill-window score (prefill.cu).  The window's queries and the pool are read through
// tensor maps; lse is [B, Hq, alpha] natural-log, scores [B, Hkv, score_stride].
struct PrefillArgs {
  CUtensorMap tmap_k;            // the K pool as [NB*Hkv*16, D] bf16, box 64 x 16, 128-byte swizzle
  CUtensorMap tmap_q;            // q_win as [B*alpha, Hq, D] bf16, box 64 x G x R, 128-byte swizzle
  const __nv_bfloat16* q_win;    // [B, alpha, Hq, D]: row r is the query of position L_b - alpha + r
  const int32_t* block_tables;   // [B, MB]
  const int32_t* context_lens;   // [B] prompt lengths
  float* lse;                    // [B, Hq, alpha]
  float* scores;                 // [B, Hkv, score_stride], added into
  int32_t* err;
  int score_stride;
  int B, Hq, Hkv, NB, MB, alpha, G;
  int R;                         // window rows per query chunk (G * R <= 64 columns)
  float scale_log2;              // scale * log2(e)
  unsigned long long timeout_ns;
};
// tcgen05 prefill-score shape: 128-key halves per CTA, window columns per chunk (the MMA's N),
// query chunks in flight, accumulators per key half, CTAs per SM the registers must allow
#ifndef PKV_TC_KH
#define PKV_TC_KH 1
#endif
#ifndef PKV_TC_COLS
#define PKV_TC_COLS 128
#endif
#ifndef PKV_TC_QSLOTS
#define PKV_TC_QSLOTS 2
#endif
#ifndef PKV_TC_ACC
#define PKV_TC_ACC 2
#endif
#ifndef PKV_TC_MINB
#define PKV_TC_MINB 2
#endif
#ifndef PKV_PREFILL_TCGEN05
#define PKV_PREFILL_TCGEN05 1  // prefill score on tcgen05 where supported (d = 128, G a power of two)
#endif
constexpr int kPrefillMaxColumns = 16384;  // alpha * G bound (the score kernel stages every lse)
constexpr int kPrefillMaxBlocks = 32768;   // block-table width bound (the lse kernel stages a row)
size_t prefill_score_smem_bytes(int head_dim, int alpha, int group);
size_t prefill_lse_smem_bytes(int head_dim, int max_blocks);
cudaError_t prefill_device_setup();
cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, bool lse_given, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialisation (it may start before the previous
// kernel on the stream ends; every kernel of this library waits for it before touching
// global memory).
inline cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

// Workspace of a decode call with partial slots for `ranges` ranges (api.cu).
struct WorkspacePlan {
  size_t ctrl_off, layout_off, ml_off, o_off, total;
  long long ranges;
};
WorkspacePlan plan_workspace(const struct pkv_dims* d, long long ranges);
WorkspacePlan fit_workspace(const struct pkv_dims* d, size_t bytes);

// Validates a paged (sparse == false) or sparse decode call, sizes its partition and
// launches it with `workspace` as scratch.  Defined in api.cu; returns a PKV status.
// Score emission of a dense decode (pkv_paged_decode_attention_scores); nullptr: none.
struct ScoreOutputs {
  float* lse;
  float* scores;
  float* logits;
  int stride;
};

// INT8 pools of a dense decode (pkv_paged_decode_attention_q8); nullptr: bf16 pools.
struct Q8Scales {
  const float* k_scale;
  const float* v_scale;
};

int decode_common(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, const int32_t* kept,
                  const int32_t* kept_lens, int32_t max_kept, float scale, int32_t window,
                  void* workspace, size_t workspace_bytes, const struct pkv_dims* dims, int32_t* err,
                  void* stream, bool sparse, const void* k_new = nullptr, const void* v_new = nullptr,
                  const ScoreOutputs* score_out = nullptr, const Q8Scales* q8 = nullptr,
                  uint32_t flags = 0);

}  // namespace pkv
