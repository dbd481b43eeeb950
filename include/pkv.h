/*
 * pkv.h -- C ABI of the paged KV-cache decode-attention library for GB300 (sm_103a).
 *
 * One decode step of an LLM attends one new query token per sequence to all of that
 * sequence's cached keys and values.  The cache is paged: K and V live in fixed-size
 * blocks of 16 tokens, and a per-sequence block table maps logical block i of a
 * sequence to a physical block anywhere in a shared pool ("KV Cache primer",
 * cf-1.com/news/5988169, section 4.1 "PagedAttention"; vLLM's --block-size 16 in
 * section 5.2).  The layer-wise sparse variant ("How KV Sparsity Achieves 1.5x
 * Acceleration for vLLM", blogs.novita.ai, sections "System model" and "Key technique 1")
 * keeps only sink tokens, a recent window and the top-scored tokens of a layer.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument that names tensor data is a DEVICE pointer owned by the
 *    caller.  The library never allocates, frees or keeps a pointer after a call returns.
 *  - Calls are asynchronous: they only enqueue kernels on `stream` (a cudaStream_t passed
 *    as void*; NULL = the legacy default stream) and never synchronise, except
 *    pkv_read_error.  The first call on a device performs one-time per-device set-up
 *    (kernel attributes, SM count); make it before capturing a stream into a CUDA graph.
 *  - Element types: K, V, q, out are bf16 (IEEE binary16-bfloat, 2 bytes); block tables,
 *    lengths and index lists are int32; slot mappings are int64.
 *  - Layouts are dense row-major with the shapes stated per argument (no strides).
 *  - Paged pool layout: k_cache and v_cache are [num_blocks, num_kv_heads, 16, head_dim];
 *    token `off` of physical block `p` for kv head `g` is row ((p*Hkv + g)*16 + off).
 *    One (block, kv-head) tile is 16*head_dim*2 bytes and contiguous (4 KiB at d=128).
 *  - A slot is a physical token position: slot = p*16 + off.  Slot < 0 means "skip".
 *  - GQA: query head h reads kv head h / G, G = num_q_heads / num_kv_heads.
 *  - Return value: PKV_OK (0) on success; a negative PKV_ERR_* for an argument the host
 *    rejects (nothing is enqueued then); PKV_ERR_CUDA_BASE + cudaError_t (>= 1000) if a
 *    launch failed.
 *  - Errors only the device can see (a block id outside the pool, a kept index outside
 *    the context, a slot outside the pool, a TMA wait that timed out) never trap: the
 *    offending access is skipped and the first such PKV_DEV_* code is stored into
 *    *error_word (a device int32 the caller zero-initialises; NULL disables reporting).
 *    Output rows touched by a device-detected error are unspecified but finite-safe.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_BLOCK_SIZE 16

/* Host-side status codes. */
#define PKV_OK 0
#define PKV_ERR_NULL_POINTER (-1)   /* a required pointer is NULL */
#define PKV_ERR_DIMS (-2)           /* a size is negative/zero where it must be positive */
#define PKV_ERR_BLOCK_SIZE (-3)     /* block_size != 16 */
#define PKV_ERR_HEAD_DIM (-4)       /* head_dim not in {64, 128} */
#define PKV_ERR_GQA (-5)            /* num_q_heads % num_kv_heads != 0 or G = Hq/Hkv > 8 */
#define PKV_ERR_WORKSPACE (-6)      /* workspace NULL or too small (see pkv_decode_workspace_bytes) */
#define PKV_ERR_ALIGNMENT (-7)      /* a tensor pointer is not 16-byte aligned */
#define PKV_ERR_ARGUMENT (-8)       /* any other invalid scalar argument */
#define PKV_ERR_NO_DEVICE (-9)      /* no current CUDA device could be queried */
#define PKV_ERR_CUDA_BASE 1000      /* + cudaError_t of a failed launch */

/* Device-side error codes stored into *error_word (first one wins). */
#define PKV_DEV_OK 0
#define PKV_DEV_BAD_BLOCK_ID 1      /* block table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_SLOT 2          /* slot >= num_blocks*16 */
#define PKV_DEV_BAD_KEPT_INDEX 3    /* kept index outside [0, context_len), or not above the one before */
#define PKV_DEV_BAD_CONTEXT_LEN 4   /* context_len < 0 or > max_blocks_per_seq*16 */
#define PKV_DEV_WAIT_TIMEOUT 5      /* an mbarrier wait exceeded its bound (kernel gave up) */
#define PKV_DEV_BAD_SCORE 6         /* NaN score given to top-k selection */
#define PKV_DEV_DIRTY_WORKSPACE 7   /* decode workspace counters were not zero at the call */
#define PKV_DEV_BAD_VALUE 8         /* non-finite K/V element given to the INT8 append */

/*
 * Flags of the decode calls (their `flags` argument; 0 = none).
 *
 * PKV_DECODE_INPUTS_READY -- the caller declares that this call's K/V pools (for INT8 pools
 *   also their scales), block_tables, context_lens and, in the sparse forms,
 *   kept_index_lists and kept_lens are not written by the work that precedes the call on
 *   its stream and may still be running when the call's first kernel starts.  With
 *   programmatic dependent launch that is the kernel enqueued just before the call and
 *   whatever that kernel lets run alongside it; when it is the previous decode call of
 *   this library, it is that call's own kernels (so the flag is wrong when that call
 *   appended into a pool this call reads).  The decode then works out its partition,
 *   fetches its first block-table entries and starts its first K/V tile copies before
 *   that work has ended, and waits for it only before it reads q, k_new/v_new, the
 *   workspace or error_word -- which the preceding kernel may therefore still produce.
 *   This is the case of a decode step's consecutive layers, each with its own pools
 *   ("KV Cache primer", cf-1.com/news/5988169, section 2.2: the step appends the new
 *   token's K/V and reads the whole cache, so every input but the new token's q, k and v
 *   is ready before the step starts).  Results are identical with and without the flag.
 * Unknown flag bits are refused with PKV_ERR_ARGUMENT.
 */
#define PKV_DECODE_INPUTS_READY 1

/*
 * Flags of pkv_kv_select_topk (its `flags` argument; 0 = none).
 *
 * PKV_SELECT_INPUTS_READY -- the caller declares that this call's score_accum and
 *   context_lens are not written by the work that precedes the call on its stream and may
 *   still be running when the call's kernel starts (with programmatic dependent launch, the
 *   kernel enqueued just before the call and whatever that kernel lets run alongside it).
 *   The selection then loads and counts its scores before that work has ended, and waits for
 *   it only before it writes kept_out, kept_lens_out or error_word -- which the preceding
 *   kernel may therefore still read or write.  This is the case of the selections of a
 *   model's layers made one after another, each from its own layer's final scores ("How KV
 *   Sparsity...", section "2. Attention modification": the scores of a layer and head are
 *   accumulated first, the top-k taken after).  Results are identical with and without the
 *   flag.  Unknown flag bits are refused with PKV_ERR_ARGUMENT.
 */
#define PKV_SELECT_INPUTS_READY 1

/*
 * Flags of pkv_kv_compact and pkv_kv_compact_q8 (their `flags` argument; 0 = none).
 *
 * PKV_COMPACT_INPUTS_READY -- the caller declares that this call's source pools (for INT8 also
 *   their scales), src_block_tables, context_lens, kept_index_lists, kept_lens and
 *   dst_block_tables are not written by the work that precedes the call on its stream and may
 *   still be running when the call's kernel starts (with programmatic dependent launch, the
 *   kernel enqueued just before the call and whatever that kernel lets run alongside it).  The
 *   compaction then reads all of them, the kept rows included, before that work has ended, and
 *   waits for it only before it writes the destination pools or error_word -- which the
 *   preceding kernel may therefore still read or write.  This is the case of the compactions of
 *   a model's sparse layers made one after another, each from its own pool through kept lists
 *   that are already final ("How KV Sparsity...", section "Key technique 1": every layer gets its
 *   own compact block table).  The first compaction after the selections that wrote the kept
 *   lists is made without the flag: a flagged selection lets the selections before it run
 *   alongside it, so the lists may still be in flight when it is the preceding work.  Results
 *   are identical with and without the flag.  Unknown flag bits are refused with
 *   PKV_ERR_ARGUMENT.
 */
#define PKV_COMPACT_INPUTS_READY 1

/*
 * Flags of pkv_kv_rolling_admit and pkv_kv_rolling_admit_q8 (their `flags` argument; 0 = none).
 *
 * PKV_ADMIT_INPUTS_READY -- the caller declares that this call's slot_pos, slot_score,
 *   kept_lens, context_lens and block_tables are not written by the work that precedes the call
 *   on its stream and may still be running when the call's kernel starts (with programmatic
 *   dependent launch, the kernel enqueued just before the call and whatever that kernel lets run
 *   alongside it).  The admission then scans the slots and chooses each (sequence, kv head)'s
 *   slot before that work has ended, and waits for it only before it reads k_new and v_new and
 *   before any write (the pool, the slot state, kept_lens, error_word) -- so the preceding
 *   kernel may still produce k_new / v_new.  This is the case of a decode step's sparse layers:
 *   a layer's slot scores were last updated by its own score pass of the previous step, and
 *   only the new token's K and V come from the work just before ("How KV Sparsity...",
 *   section "System model").  Results are identical with and without the flag.  Unknown flag
 *   bits are refused with PKV_ERR_ARGUMENT.
 */
#define PKV_ADMIT_INPUTS_READY 1

/* Shape record shared by the calls. */
typedef struct pkv_dims {
  int32_t batch;              /* B: sequences in this decode step */
  int32_t num_q_heads;        /* Hq */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0 */
  int32_t head_dim;           /* d: 64 or 128 */
  int32_t block_size;         /* tokens per physical block; must be 16 */
  int32_t num_blocks;         /* NB: physical blocks in each of the K and V pools */
  int32_t max_blocks_per_seq; /* MB: row length of block_tables */
} pkv_dims;

/*
 * pkv_kv_append -- write this step's new key/value rows into their cache slots.
 * Defines: the decode stage computes K,V of the new token only and appends them to the
 * cache ("KV Cache primer", cf-1.com/news/5988169, section 2.2); all layers of one step
 * share one write position ("naive KV cache", koas-w.github.io/posts/20260325-kvcache,
 * the seq_len pitfall), so one slot_mapping serves every layer.
 *   k_cache, v_cache : [NB, Hkv, 16, d] bf16, updated in place.
 *   k, v             : [num_tokens, Hkv, d] bf16, the new rows.
 *   slot_mapping     : [num_tokens] int64; token i goes to slot slot_mapping[i]
 *                      (block slot/16, offset slot%16) for every kv head; < 0 skips it.
 *                      Two tokens with the same slot in one call is invalid input.
 *   num_tokens       : >= 0 (0 enqueues nothing).
 *   dims             : uses num_kv_heads, head_dim, block_size, num_blocks.
 *   error_word       : optional; receives PKV_DEV_BAD_SLOT for slot >= NB*16.
 * Bit-exact: the cache rows become exactly the input bits.
 */
int pkv_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                  const int64_t* slot_mapping, int64_t num_tokens, const pkv_dims* dims,
                  int32_t* error_word, void* stream);

/*
 * pkv_decode_workspace_bytes -- bytes of device workspace for pkv_paged_decode_attention and
 * pkv_paged_decode_attention_append with these dims.  The split-K decode cuts the work into
 * one slice per worker warp (at most 2048 warps): a static head per warp plus up to four
 * tail chunks per slice that warps take from a ticket counter as they finish, and keeps two
 * partial results per such range: about 2 * 10240 * G * (d + 2) * 4 bytes, whatever the
 * context lengths (G = Hq / Hkv).  A smaller workspace is accepted as long as it holds the
 * partials of 2048 ranges; it then gets fewer tail chunks.
 * The workspace's first 8 bytes are the ticket counters: they must be zero before the
 * first call (e.g. allocate it zero-filled) and every call leaves them zero, so one
 * workspace serves consecutive calls on one stream, of any shape, without re-clearing.
 * Counters found non-zero make the call record PKV_DEV_DIRTY_WORKSPACE.
 * Returns 0 if dims are invalid.
 */
size_t pkv_decode_workspace_bytes(const pkv_dims* dims);

/*
 * pkv_paged_decode_attention -- out = softmax(scale * q K^T) V per sequence and query head.
 * Defines: the attention formula ("Transformer模型中的KV Cache优化推理策略",
 * yutianautomatic.com, section "为什么传统推理方式难以为继"), evaluated at decode time
 * with the new token's query against all cached keys ("KV Cache primer" section 2.2), K/V
 * gathered through the block table (section 4.1); the optional sliding window keeps only
 * the most recent `window` tokens (section 4.3).  Computed with the one-pass online softmax
 * (running max and running sum, output divided by the sum at the end) of "How KV Sparsity
 * Achieves 1.5x Acceleration for vLLM", section "2. Attention modification" (Fig. 7),
 * split over context blocks and merged by log-sum-exp.
 *   out            : [B, Hq, d] bf16 (round-to-nearest-even of the fp32 result).
 *   q              : [B, Hq, d] bf16.
 *   k_cache,v_cache: [NB, Hkv, 16, d] bf16.
 *   block_tables   : [B, MB] int32; entry [b][i] = physical block of logical block i.
 *                    Only the entries covering the attended tokens are read.
 *   context_lens   : [B] int32; L_b = tokens of sequence b INCLUDING this step's token;
 *                    0 <= L_b <= MB*16.  L_b == 0 gives a zero output row.
 *   scale          : logit scale (normally 1/sqrt(d)).
 *   window         : > 0 attends tokens [max(0, L_b - window), L_b); <= 0 attends all.
 *   workspace      : pkv_decode_workspace_bytes(dims) bytes, 16-byte aligned, its first 8
 *                    bytes zero before the first use (every call leaves them zero).
 *   flags          : 0 or PKV_DECODE_INPUTS_READY (see there); the same in every decode call.
 *   error_word     : optional; PKV_DEV_BAD_BLOCK_ID / _BAD_CONTEXT_LEN / _WAIT_TIMEOUT /
 *                    _DIRTY_WORKSPACE.
 * Supported: d in {64, 128}; G = Hq / Hkv in 1..8.
 */
int pkv_paged_decode_attention(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, float scale, int32_t window,
                               void* workspace, size_t workspace_bytes, const pkv_dims* dims,
                               uint32_t flags, int32_t* error_word, void* stream);

/*
 * pkv_paged_decode_attention_append -- one decode step's KV append and attention in one
 * kernel: the same result as pkv_kv_append of this step's token followed by
 * pkv_paged_decode_attention, for the usual decode layout in which the new token of
 * sequence b is its logical position L_b - 1 (L_b = context_lens[b] counts it).  The step's
 * K/V rows are written into the pool at that position (block block_tables[b][(L_b-1)/16],
 * offset (L_b-1)%16, every kv head) and used for it directly, which saves the separate
 * append launch and the re-read of the freshly written rows ("KV Cache primer",
 * cf-1.com/news/5988169, section 2.2: compute the new token's K,V, append, attend).
 *   k_cache, v_cache : [NB, Hkv, 16, d] bf16, read and updated in place.
 *   k_new, v_new     : [B, Hkv, d] bf16, the step's new rows (one token per sequence).
 *   other arguments  : as pkv_paged_decode_attention; sequences with L_b == 0 append nothing.
 */
int pkv_paged_decode_attention_append(void* out, const void* q, void* k_cache, void* v_cache,
                                      const void* k_new, const void* v_new,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      float scale, int32_t window, void* workspace,
                                      size_t workspace_bytes, const pkv_dims* dims,
                                      uint32_t flags, int32_t* error_word, void* stream);

/*
 * INT8 KV cache: K and V stored as 8-bit integers, which halves the cache ("KV Cache
 * primer", cf-1.com/news/5988169, section 4.2; section 5.2 enables it in vLLM with
 * --kv-cache-dtype int8).  The pages give no scheme; the one used here is symmetric absmax
 * quantization per (token, kv head) row: scale s = max|x| / 127 (fp32), codes
 * c = round_half_even(x / s) clamped to [-127, 127] (single-precision IEEE division and
 * rounding), value c * s.  A zero row has s = 0 and codes 0.
 * Code pools are [NB, Hkv, 16, d] uint8 (the bf16 layout, one byte per element) holding each
 * code c as the byte c + 128 (1..255 for the codes this rule makes; a byte b is read as the
 * code b - 128); scale pools are [NB, Hkv, 16] fp32 (one scale per row: 4/d bytes per element
 * more, 3.1 % at d = 128).
 *
 * pkv_kv_append_q8 -- pkv_kv_append into INT8 pools: each new K and V row is quantized into
 * its slot.
 *   k_codes, v_codes   : [NB, Hkv, 16, d] uint8, updated in place.
 *   k_scales, v_scales : [NB, Hkv, 16] fp32, updated in place.
 *   k, v, slot_mapping, num_tokens, dims : as pkv_kv_append.
 *   error_word         : optional; PKV_DEV_BAD_SLOT, or PKV_DEV_BAD_VALUE for a token whose K or
 *                        V row holds a non-finite value (its rows are then left unwritten).
 * All pointers 16-byte aligned.  Bit-exact: the codes and scales of the rule above.
 */
int pkv_kv_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k,
                     const void* v, const int64_t* slot_mapping, int64_t num_tokens, const pkv_dims* dims,
                     int32_t* error_word, void* stream);

/*
 * pkv_paged_decode_attention_q8 -- pkv_paged_decode_attention over INT8 pools: every K and V
 * element is read as code * scale of its row.  Reads half the K/V bytes (plus the scales).
 *   k_codes, v_codes   : [NB, Hkv, 16, d] uint8.
 *   k_scales, v_scales : [NB, Hkv, 16] fp32, 16-byte aligned; rows of tokens outside the
 *                        attended set are never used.
 *   other arguments    : as pkv_paged_decode_attention; the same workspace
 *                        (pkv_decode_workspace_bytes) serves both.
 * Computed with fp16 tensor-core products of the exact codes and of q scaled by a power of
 * two into fp16 range (exact for bf16 q), fp32 sums; the row scales are applied in fp32.
 */
int pkv_paged_decode_attention_q8(void* out, const void* q, const void* k_codes, const void* v_codes,
                                  const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                  const int32_t* context_lens, float scale, int32_t window, void* workspace,
                                  size_t workspace_bytes, const pkv_dims* dims, uint32_t flags,
                                  int32_t* error_word,
                                  void* stream);

/*
 * pkv_paged_decode_attention_append_q8 -- pkv_kv_append_q8 fused into
 * pkv_paged_decode_attention_q8 for the usual decode slot, as pkv_paged_decode_attention_append
 * does for bf16 pools: each sequence's new token is at position L_b - 1 (its slot comes from
 * the block table), its K and V rows are quantized by the row rule of pkv_kv_append_q8 into the
 * code and scale pools, and the decode attends over them.
 *   k_codes, v_codes, k_scales, v_scales : INT8 pools as pkv_paged_decode_attention_q8, updated
 *                        in place at each sequence's position L_b - 1 (L_b >= 1).
 *   k_new, v_new       : [B, Hkv, d] bf16, 16-byte aligned.
 *   other arguments    : as pkv_paged_decode_attention_q8.
 *   error_word         : as pkv_paged_decode_attention_q8, plus PKV_DEV_BAD_VALUE when a new row
 *                        holds a non-finite value (that (b, kv head)'s rows are then not written
 *                        and its attention reads the pool as it was).
 * The pools end bit-identical to pkv_kv_append_q8 of the same rows, and out bit-identical to
 * pkv_paged_decode_attention_q8 over the appended pools (same workspace size).
 */
int pkv_paged_decode_attention_append_q8(void* out, const void* q, void* k_codes, void* v_codes, float* k_scales,
                                         float* v_scales, const void* k_new, const void* v_new,
                                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                                         int32_t window, void* workspace, size_t workspace_bytes,
                                         const pkv_dims* dims, uint32_t flags, int32_t* error_word,
                                         void* stream);

/*
 * pkv_prefill_window_scores -- the prefill-side sparsification score: after a prompt of L_b
 * tokens, key i of kv head g scores the sum, over the last alpha prompt positions j (the
 * instruction window, j >= i) and the G query heads of the group, of its causal softmax
 * probability exp(scale * q_j . k_i - lse_j) ("How KV Sparsity Achieves 1.5x Acceleration for
 * vLLM", section "2. Attention modification": the PyramidKV score computed from the forward
 * pass's rowmax and l, with the loop over keys outermost).  The sums are ADDED into
 * score_accum, which then feeds pkv_kv_select_topk.
 *   score_accum  : [B, Hkv, score_stride] fp32, 4-byte aligned; keys >= score_stride get no score
 *                  (PKV_DEV_BAD_CONTEXT_LEN is recorded).
 *   lse          : [B, Hq, alpha] fp32 natural-log row log-sum-exps of the window rows.  With
 *                  lse_given != 0 they are read (the prefill attention's rowmax + log l); with
 *                  lse_given == 0 they are computed first (a pass over each row's causal keys)
 *                  and written; rows of negative position (L_b < alpha) get -infinity.
 *   q_win        : [B, alpha, Hq, d] bf16, 16-byte aligned; row r is the query of position
 *                  L_b - alpha + r (rows of negative position are not read).
 *   k_cache      : [NB, Hkv, 16, d] bf16 pool; block_tables [B, MB]; context_lens [B] = L_b.
 *   alpha        : >= 1, alpha * G <= 16384.     scale : logit scale.
 *   error_word   : optional; PKV_DEV_BAD_BLOCK_ID, _BAD_CONTEXT_LEN, _WAIT_TIMEOUT.
 * Supported: d in {64, 128}; G = Hq / Hkv in 1..8; MB <= 32768 blocks.
 */
int pkv_prefill_window_scores(float* score_accum, int32_t score_stride, float* lse, int32_t lse_given,
                              const void* q_win, const void* k_cache, const int32_t* block_tables,
                              const int32_t* context_lens, int32_t alpha, float scale, const pkv_dims* dims,
                              int32_t* error_word, void* stream);

/*
 * pkv_paged_decode_attention_scores -- pkv_paged_decode_attention (with this step's append
 * when k_new and v_new are given, as pkv_paged_decode_attention_append) that also produces
 * the step's sparsification score: the scoring of "How KV Sparsity Achieves 1.5x
 * Acceleration for vLLM", section "2. Attention modification" -- the attention pass already
 * has each row's maximum and normaliser (rowmax / l), so every attended key's softmax
 * probability is exp(s - rowmax) / l, and a key's score is the sum of such probabilities.
 * A kv head's key serves the G query heads of its group, so its score adds their G
 * probabilities.  The pages' kernel recomputes q . k in a second pass; here the decode keeps
 * every attended key's logit (4 bytes per query head and key) and a light second kernel
 * turns them into probabilities, which reads far fewer bytes than reading K again.
 *   lse_out        : [B, Hq] fp32: natural log-sum-exp of each row's attended logits
 *                    (-infinity when nothing is attended).
 *   score_accum    : [B, Hkv, score_stride] fp32, updated in place: for every attended
 *                    position t < score_stride of (b, kv head g),
 *                    score_accum[b][g][t] += sum over h in g's group of p_{b,h,t}.
 *                    Other positions are left unchanged.
 *   logits         : [B, Hq, score_stride] fp32 scratch, caller-owned; contents on return
 *                    unspecified.
 *   score_stride   : > 0; should be >= every L_b (max_blocks_per_seq * 16 always is): keys
 *                    at positions >= score_stride get no score and the call records
 *                    PKV_DEV_BAD_CONTEXT_LEN.
 *   k_new, v_new   : both NULL (no append) or both set, as pkv_paged_decode_attention_append.
 *   other arguments: as pkv_paged_decode_attention.  out is bit-identical to what that call
 *                    (or the append variant) writes for the same inputs and workspace size.
 * Same device error codes as pkv_paged_decode_attention.
 */
int pkv_paged_decode_attention_scores(void* out, float* lse_out, float* score_accum, float* logits,
                                      int32_t score_stride, const void* q, void* k_cache,
                                      void* v_cache, const void* k_new, const void* v_new,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      float scale, int32_t window, void* workspace,
                                      size_t workspace_bytes, const pkv_dims* dims,
                                      uint32_t flags, int32_t* error_word, void* stream);

/*
 * pkv_paged_decode_attention_scores_q8 -- pkv_paged_decode_attention_scores over INT8 pools
 * (no append: INT8 pools take this step's token through pkv_kv_append_q8 first).  Every K
 * element is read as code * scale of its row for the logits, every V element likewise for the
 * output, as pkv_paged_decode_attention_q8; the score, lse and logits outputs are those of
 * pkv_paged_decode_attention_scores for the dequantized K.
 *   k_codes, v_codes, k_scales, v_scales : as pkv_paged_decode_attention_q8.
 *   other arguments : as pkv_paged_decode_attention_scores.  out is bit-identical to what
 *                     pkv_paged_decode_attention_q8 writes for the same inputs and workspace size.
 */
int pkv_paged_decode_attention_scores_q8(void* out, float* lse_out, float* score_accum, float* logits,
                                         int32_t score_stride, const void* q, const void* k_codes,
                                         const void* v_codes, const float* k_scales, const float* v_scales,
                                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                                         int32_t window, void* workspace, size_t workspace_bytes,
                                         const pkv_dims* dims, uint32_t flags, int32_t* error_word,
                                         void* stream);

/*
 * pkv_sparse_decode_workspace_bytes -- workspace for pkv_sparse_decode_attention with
 * kept lists of row length max_kept: the same size and rules as pkv_decode_workspace_bytes
 * (it does not depend on max_kept).  Returns 0 if the arguments are invalid.
 */
size_t pkv_sparse_decode_workspace_bytes(const pkv_dims* dims, int32_t max_kept);

/*
 * pkv_sparse_decode_attention -- decode attention over a kept subset of each sequence's
 * tokens (the layer-wise sparse variant: a layer keeps high-score and recent KV and drops
 * the rest, "How KV Sparsity Achieves 1.5x Acceleration for vLLM", sections "System
 * model" and "Key technique 1").  Same formula as pkv_paged_decode_attention, with the
 * attended set of (b, kv head g) = kept_index_lists[b][g][0 : kept_lens[b]], gathered row
 * by row from the full paged pool through block_tables.
 *   kept_index_lists : [B, Hkv, max_kept] int32 logical token positions, strictly
 *                      ascending, each in [0, context_lens[b]).  An entry outside that range
 *                      or not above the entry before it (a duplicate or a descent) is reported
 *                      as PKV_DEV_BAD_KEPT_INDEX and not attended; that (b, kv head)'s rows are
 *                      then unspecified, every other row is unaffected.
 *   kept_lens        : [B] int32 in [0, max_kept]; every kv head of b keeps that many.
 *   other arguments  : as pkv_paged_decode_attention (no window).
 */
int pkv_sparse_decode_attention(void* out, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens,
                                const int32_t* kept_index_lists, const int32_t* kept_lens,
                                int32_t max_kept, float scale, void* workspace,
                                size_t workspace_bytes, const pkv_dims* dims,
                                uint32_t flags, int32_t* error_word, void* stream);

/*
 * pkv_kv_select_topk -- choose the tokens a sparse layer keeps, per (sequence, kv head):
 * the first n_sink tokens (attention sinks: the start token carries massive activations,
 * "How KV Sparsity..." introduction, Fig. 1), the n_recent most recent tokens, and the
 * k_top highest-scoring tokens among the rest (pruning drops low-score KV pairs and
 * retains high-score and nearby ones, section "System model"; the score is per layer and
 * head, a sum of softmax probabilities, section "2. Attention modification").
 *   kept_out       : [B, Hkv, n_sink + k_top + n_recent] int32, ascending token positions;
 *                    entries past kept_lens_out[b] are left untouched.
 *   kept_lens_out  : [B] int32 = min(L_b, n_sink + k_top + n_recent).
 *   score_accum    : [B, Hkv, score_stride] fp32; score of token t is [b][g][t], t < L_b.
 *   context_lens   : [B] int32, 0 <= L_b <= score_stride.
 * Rule: if L_b <= n_sink + k_top + n_recent every token is kept.  Otherwise candidates are
 * [n_sink, L_b - n_recent), ordered by score descending, equal scores by lower position
 * first (-0.0 equals +0.0); the first k_top candidates are kept.  Bit-exact.  NaN scores are
 * invalid (PKV_DEV_BAD_SCORE).  Supports score_stride <= 262144.
 *   flags          : 0 or PKV_SELECT_INPUTS_READY (see there).
 */
int pkv_kv_select_topk(int32_t* kept_out, int32_t* kept_lens_out, const float* score_accum,
                       int32_t score_stride, const int32_t* context_lens, int32_t n_sink,
                       int32_t n_recent, int32_t k_top, const pkv_dims* dims, uint32_t flags,
                       int32_t* error_word, void* stream);

/*
 * pkv_kv_compact -- copy each (sequence, kv head)'s kept tokens into a compact paged pool:
 * compact position j of (b, g) receives source token kept_index_lists[b][g][j], so that
 * the compact pool holds the layer's retained KV in 16-token blocks and plain paged decode
 * over it with context length kept_lens[b] equals sparse decode over the full pool (the
 * per-layer block-table policy of "How KV Sparsity...", section "Key technique 1", Fig. 5).
 *   dst_k_cache, dst_v_cache : [dst_num_blocks, Hkv, 16, d] bf16, written at the slots the
 *                              copy addresses; other slots untouched.
 *   dst_block_tables         : [B, dst_max_blocks_per_seq] int32.
 *   src_*                    : the full pool and its block table, shapes per src_dims.
 *   context_lens             : [B] int32 source context lengths (for index validation).
 *   kept_index_lists, kept_lens, max_kept : as pkv_sparse_decode_attention; an entry outside
 *                              [0, L_b) or not above the one before it is reported
 *                              (PKV_DEV_BAD_KEPT_INDEX) and its compact slot left untouched.
 *   flags                    : 0 or PKV_COMPACT_INPUTS_READY (see there).
 * Bit-exact.
 */
int pkv_kv_compact(void* dst_k_cache, void* dst_v_cache, const int32_t* dst_block_tables,
                   int32_t dst_num_blocks, int32_t dst_max_blocks_per_seq,
                   const void* src_k_cache, const void* src_v_cache,
                   const int32_t* src_block_tables, const int32_t* context_lens,
                   const int32_t* kept_index_lists, const int32_t* kept_lens,
                   int32_t max_kept, const pkv_dims* src_dims, uint32_t flags,
                   int32_t* error_word, void* stream);

/*
 * pkv_sparse_decode_attention_q8 -- pkv_sparse_decode_attention over INT8 pools: the attended set
 * of (b, kv head g) is its kept list, and every K and V element is read as code * scale of its
 * row (the arithmetic of pkv_paged_decode_attention_q8).  Rows are gathered through the kept
 * lists (the codes as 16-byte asynchronous copies, the two row scales as 4-byte ones).
 *   k_codes, v_codes, k_scales, v_scales : as pkv_paged_decode_attention_q8.
 *   other arguments    : as pkv_sparse_decode_attention (same workspace, same errors).
 */
int pkv_sparse_decode_attention_q8(void* out, const void* q, const void* k_codes, const void* v_codes,
                                   const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                   const int32_t* context_lens, const int32_t* kept_index_lists,
                                   const int32_t* kept_lens, int32_t max_kept, float scale, void* workspace,
                                   size_t workspace_bytes, const pkv_dims* dims, uint32_t flags,
                                   int32_t* error_word, void* stream);

/*
 * pkv_kv_compact_q8 -- pkv_kv_compact over INT8 pools: each kept row's codes and its fp32 row
 * scale move together, so the compact pool holds the same values (code * scale).
 *   dst_k_codes, dst_v_codes, src_k_codes, src_v_codes : [NB, Hkv, 16, d] uint8 pools.
 *   dst_k_scales, dst_v_scales, src_k_scales, src_v_scales : [NB, Hkv, 16] fp32 row scales.
 *   other arguments : as pkv_kv_compact.  All pool pointers 16-byte aligned.  Bit-exact.
 */
int pkv_kv_compact_q8(void* dst_k_codes, void* dst_v_codes, float* dst_k_scales, float* dst_v_scales,
                      const int32_t* dst_block_tables, int32_t dst_num_blocks, int32_t dst_max_blocks_per_seq,
                      const void* src_k_codes, const void* src_v_codes, const float* src_k_scales,
                      const float* src_v_scales, const int32_t* src_block_tables, const int32_t* context_lens,
                      const int32_t* kept_index_lists, const int32_t* kept_lens, int32_t max_kept,
                      const pkv_dims* src_dims, uint32_t flags, int32_t* error_word, void* stream);

/*
 * pkv_kv_rolling_admit -- admit one decode step's token into each sequence's sparse-layer cache
 * of fixed budget: capacity = n_sink + k_top + n_recent slots per (sequence, kv head) in a
 * compact pool (slot s at block block_tables[b][s / 16], offset s % 16).  The rolling form of
 * the layer-wise sparse cache of "How KV Sparsity Achieves 1.5x Acceleration for vLLM"
 * (section "System model": a sparse layer keeps high-score and recent KV; the new KV replaces
 * the lowest-score KV).  Per (b, kv head g):
 *   - kept_lens[b] < capacity: the token takes slot kept_lens[b];
 *   - full: the token at position L_b - 1 - n_recent leaves the recent window and meets the
 *     top-k set (the slots holding positions in [n_sink, L_b - 1 - n_recent)): if its score is
 *     strictly greater than the set's lowest score (among equal lowest scores the highest
 *     position is the weakest), the weakest is dropped, otherwise the leaving token is; the
 *     new token takes the dropped token's slot.  Sinks and the recent window are never dropped.
 * The slot taken receives k_new[b][g] / v_new[b][g], position L_b - 1 and score 0;
 * kept_lens[b] grows by one while below capacity.  Bit-exact.
 *   k_cache, v_cache : compact pool [NB, Hkv, 16, d] bf16, updated in place.
 *   block_tables     : [B, MB] int32 compact tables; capacity <= MB * 16.
 *   slot_pos         : [B, Hkv, capacity] int32 logical positions held (updated).
 *   slot_score       : [B, Hkv, capacity] fp32 accumulated scores (updated), e.g. from
 *                      pkv_paged_decode_attention_scores over the compact pool.
 *   kept_lens        : [B] int32 slots in use (updated).
 *   context_lens     : [B] int32 L_b counting the new token (>= 1).
 *   k_new, v_new     : [B, Hkv, d] bf16.
 *   flags            : 0 or PKV_ADMIT_INPUTS_READY (see there).
 *   error_word       : optional; PKV_DEV_BAD_SCORE (a NaN score), PKV_DEV_BAD_KEPT_INDEX (the
 *                      leaving token is in no slot), PKV_DEV_BAD_BLOCK_ID, PKV_DEV_BAD_CONTEXT_LEN;
 *                      that (b, g) (or b) is then left unchanged.
 */
int pkv_kv_rolling_admit(void* k_cache, void* v_cache, const int32_t* block_tables,
                         int32_t* slot_pos, float* slot_score, int32_t* kept_lens,
                         const int32_t* context_lens, const void* k_new, const void* v_new,
                         int32_t capacity, int32_t n_sink, int32_t n_recent, const pkv_dims* dims,
                         uint32_t flags, int32_t* error_word, void* stream);

/*
 * pkv_kv_rolling_admit_q8 -- pkv_kv_rolling_admit into INT8 pools: the same choice of slot,
 * and the new token's K and V rows quantized into it by the row rule of pkv_kv_append_q8.
 *   k_codes, v_codes   : [NB, Hkv, 16, d] uint8 compact pools, updated in place.
 *   k_scales, v_scales : [NB, Hkv, 16] fp32 row scales, updated in place.
 *   other arguments    : as pkv_kv_rolling_admit.
 *   error_word         : as pkv_kv_rolling_admit, plus PKV_DEV_BAD_VALUE for a (b, g) whose new K
 *                        or V row holds a non-finite value (its rows, position and score are
 *                        then left unchanged).
 * All pool pointers 16-byte aligned.  Bit-exact.
 */
int pkv_kv_rolling_admit_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                            const int32_t* block_tables, int32_t* slot_pos, float* slot_score, int32_t* kept_lens,
                            const int32_t* context_lens, const void* k_new, const void* v_new, int32_t capacity,
                            int32_t n_sink, int32_t n_recent, const pkv_dims* dims, uint32_t flags,
                            int32_t* error_word, void* stream);

/*
 * pkv_paged_decode_attention_fixed_scratch -- pkv_paged_decode_attention for callers that
 * cannot allocate device memory.  It has no counterpart on the pages: it exists only for
 * callers with no device allocator at hand (for example a plain C program or plugin that
 * links just this library) or whose host runtime owns the device heap and forbids
 * cudaMalloc (which can also synchronise the device at a moment the caller cannot afford).
 * It takes the same inputs and output as pkv_paged_decode_attention minus the workspace:
 * the split-K scratch is a static device array of PKV_FIXED_SCRATCH_BYTES (16 MiB) inside
 * the library, which every GPU that loads the library keeps until the process exits.  The
 * call itself allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - It holds the partial results of 2048 worker ranges plus load-balancing chunks as
 *     far as it has room (see pkv_decode_workspace_bytes).  Shapes for which 2048 ranges
 *     do not fit -- G * d above 512, that is G = 8 at d = 128 -- return PKV_ERR_WORKSPACE
 *     and enqueue nothing.
 *   - The first call on a device looks up the array's device address on that device (with
 *     it current); make that first call before any stream capture.  The address is kept for
 *     the life of the process: a cudaDeviceReset after the first call (which reloads the
 *     library's device code) is not supported by this entry point.
 *   - Every call on a device shares the one array.  Its two control words start at zero
 *     (static storage) and every completed call leaves them zero.  If a call returns a
 *     launch error (>= PKV_ERR_CUDA_BASE) after its first kernel was enqueued, the words may
 *     be left non-zero: the next call then reports PKV_DEV_DIRTY_WORKSPACE, its result is
 *     not to be used, and it clears them, so the call after it is correct again.  Calls
 *     whose kernels overlap on the GPU -- different streams without ordering, or several
 *     host threads -- race on it and give wrong results: serialise them.
 *   - Results equal those of pkv_paged_decode_attention up to fp32 summation order (with
 *     fewer load-balancing chunks the split-K partition may differ).
 */
#define PKV_FIXED_SCRATCH_BYTES (16 * 1024 * 1024)
int pkv_paged_decode_attention_fixed_scratch(void* out, const void* q, const void* k_cache,
                                             const void* v_cache, const int32_t* block_tables,
                                             const int32_t* context_lens, float scale,
                                             int32_t window, const pkv_dims* dims,
                                             int32_t* error_word, void* stream);

/*
 * pkv_device_alias -- the device address of pinned (page-locked) host memory, for the decode
 * calls' arguments that their kernels reach with ordinary loads and stores: q, k_new, v_new,
 * block_tables, context_lens and out of every *_decode_attention* call may be pinned host
 * memory passed by this address (not the K/V pools, read through tensor maps, nor the
 * workspace, error_word or score buffers).  The kernels then read and write that memory in
 * place over the host link (NVLink-C2C on a Grace-Blackwell node), so a step's inputs need no
 * copy to the device and its output none back, and consecutive calls stay adjacent on the
 * stream.  The memory must stay pinned and unchanged by the host until the calls that use it
 * have completed.
 *   host_ptr   : an address inside memory allocated with cudaHostAlloc / cudaMallocHost (or
 *                registered with cudaHostRegister, mapped).
 *   device_ptr : receives the device address (on unified-addressing systems the same value).
 * Returns PKV_OK, PKV_ERR_NULL_POINTER, or PKV_ERR_ARGUMENT when the memory is not pinned and
 * mapped for the current device (*device_ptr is then NULL).  Host only; no device work.
 */
int pkv_device_alias(const void* host_ptr, void** device_ptr);

/*
 * pkv_read_error -- synchronise `stream`, then return the device error word's value
 * (PKV_DEV_*), or a negative host status if it cannot be read.  If `clear` is non-zero
 * the word is reset to 0 afterwards.  Diagnostic; not for the hot loop.
 */
int pkv_read_error(int32_t* error_word, int32_t clear, void* stream);

/* Human-readable text for a host status (PKV_OK / PKV_ERR_*) or >= PKV_ERR_CUDA_BASE. */
const char* pkv_status_string(int status);

/* Human-readable text for a device error code (PKV_DEV_*). */
const char* pkv_device_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
