// api.cu -- the extern "C" boundary declared in include/pkv.h: argument validation on the
// host, per-device one-time set-up, workspace sizing and kernel launches on the caller's
// stream.  Allocates nothing and never synchronises (except pkv_read_error).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxBatch = 4096;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per mbarrier wait
constexpr int kNumHeadDims = 2;
constexpr int kGroups[] = {1};  // every group size shares one kernel per (head_dim, mode)
constexpr int kNumGroups = 1;

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  size_t max_dyn_smem[2][6] = {};  // [head_dim index][mode: dense, sparse, dense + scores,
                                   //   dense INT8, INT8 + scores, sparse INT8]: opt-in minus static
                                   //   shared memory
  int merge_ctas_per_sm[2] = {};   // [head_dim index]: resident merge CTAs per SM
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

int head_dim_index(int d) { return d == 128 ? 0 : (d == 64 ? 1 : -1); }

// One-time per-device set-up: SM count and the dynamic shared-memory opt-in of every decode
// instantiation.  Not a stream operation, so it is legal while a stream is being captured,
// but the first call should still precede capture.
const DeviceInfo* device_info(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = PKV_ERR_NO_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& info = g_devices[dev];
  if (!info.ready) {
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      *status = PKV_ERR_NO_DEVICE;
      return nullptr;
    }
    for (int hd = 0; hd < kNumHeadDims; ++hd) {
      for (int gi = 0; gi < kNumGroups; ++gi) {
        for (int sp = 0; sp < 6; ++sp) {
          const DecodeKernel k =
              decode_kernel(hd == 0 ? 128 : 64, kGroups[gi], sp == 1 || sp == 5, sp == 2 || sp == 4, sp >= 3);
          if (k.split == nullptr) continue;
          cudaFuncAttributes fa{};
          cudaError_t e = cudaFuncGetAttributes(&fa, k.split);
          const int dyn = optin - (int)fa.sharedSizeBytes;
          if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k.split, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
          if (e != cudaSuccess) {
            cudaGetLastError();
            *status = PKV_ERR_CUDA_BASE + (int)e;
            return nullptr;
          }
          info.max_dyn_smem[hd][sp] = (size_t)dyn;
          int per_sm = 0;
          e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.merge, kMergeWarps * 32, 0);
          if (e != cudaSuccess) {
            cudaGetLastError();
            *status = PKV_ERR_CUDA_BASE + (int)e;
            return nullptr;
          }
          info.merge_ctas_per_sm[hd] = per_sm > 0 ? per_sm : 1;
        }
      }
    }
    {
      cudaError_t e = kvops_device_setup();
      if (e == cudaSuccess) e = prefill_device_setup();
      if (e != cudaSuccess) {
        cudaGetLastError();
        *status = PKV_ERR_CUDA_BASE + (int)e;
        return nullptr;
      }
    }
    info.sm_count = sms;
    info.ready = true;
  }
  *status = PKV_OK;
  return &info;
}

// cuTensorMapEncodeTiled, resolved once through the runtime (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  });
  return fn;
}

// A pool [NB, Hkv, 16, D] viewed as a 2-D bf16 tensor of NB*Hkv*16 rows of D elements, read
// in boxes of 64 columns (128 bytes) x 16 rows with the 128-byte swizzle.
int encode_pool_map(CUtensorMap* map, const void* base, long long rows, int head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return PKV_ERR_NO_DEVICE;
  const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                         elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_ARGUMENT;
}

// An INT8 pool [NB, Hkv, 16, D] as a 2-D byte tensor of NB*Hkv*16 rows of D bytes, read in
// one box of D bytes x 16 rows with the swizzle of the row size (128 or 64 bytes).
int encode_pool_map_q8(CUtensorMap* map, const void* base, long long rows, int head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return PKV_ERR_NO_DEVICE;
  const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)head_dim};
  const cuuint32_t box[2] = {(cuuint32_t)head_dim, 16};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                         elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_ARGUMENT;
}

// The prefill window's queries [B*alpha, Hq, D] bf16 as a 3-D tensor read in boxes of 64
// columns x G heads x R window rows (one query chunk: G*R columns of 128 bytes each).
int encode_window_map(CUtensorMap* map, const void* base, long long rows, int num_q_heads, int head_dim, int group,
                      int chunk_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return PKV_ERR_NO_DEVICE;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_q_heads * head_dim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)chunk_rows};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                         elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_ARGUMENT;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const pkv_dims* d, bool need_q_heads) {
  if (d == nullptr) return PKV_ERR_NULL_POINTER;
  if (d->block_size != PKV_BLOCK_SIZE) return PKV_ERR_BLOCK_SIZE;
  if (head_dim_index(d->head_dim) < 0) return PKV_ERR_HEAD_DIM;
  if (d->batch < 0 || d->num_kv_heads <= 0 || d->num_blocks < 0 || d->max_blocks_per_seq < 0)
    return PKV_ERR_DIMS;
  if (need_q_heads) {
    if (d->num_q_heads <= 0) return PKV_ERR_DIMS;
    if (d->num_q_heads % d->num_kv_heads != 0) return PKV_ERR_GQA;
  }
  return PKV_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA_BASE + (int)e; }

// Merge warps per output row (log2), from an upper estimate of the partials a row has: one
// more warp per PKV_MERGE_PARTIALS_PER_WARP partials, at most 8, and no more than the GPU holds
// in one wave of merge CTAs.
// The estimate mirrors the split kernel's partition with every sequence at its maximum length.
int merge_warps_log2(const pkv_dims* d, int max_units, long long workers, int min_units, int min_busy_pct,
                     int tail_pct, int chunk_min, int cpw_cap, long long resident_warps, int partials_per_warp) {
  const long long total = (long long)d->batch * d->num_kv_heads * max_units;
  long long P = (total + workers - 1) / workers;
  const long long busy = std::max(1ll, workers * min_busy_pct / 100);
  const long long floor_units = std::min<long long>(min_units, (total + busy - 1) / busy);
  if (P < floor_units) P = floor_units;
  const long long tail = P * tail_pct / 100;
  int cpw = 0;
  while (cpw < cpw_cap && tail >= chunk_min * ((2ll << cpw) - 1)) ++cpw;
  const long long np = ((long long)max_units + P - 1) / P * (1 + cpw) + 1;
  int lg = 0;
  while (lg < 3 && np >= (long long)partials_per_warp << (lg + 1)) ++lg;
  const long long rows = (long long)d->batch * d->num_q_heads;
  while (lg > 0 && (rows << lg) > resident_warps) --lg;
  return lg;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// Workspace layout of the decode calls (offsets 256-byte aligned):
//   uint32 ctrl[2] | int32 layout[2B] | float2 part_ml[2 * ranges][G] | float part_o[2 * ranges][G][D]
// for a workspace with partial slots for `ranges` ranges (two per range: its first and its
// last segment).  ctrl must be zero before the first call; every call leaves it zero.
WorkspacePlan plan_workspace(const pkv_dims* d, long long ranges) {
  WorkspacePlan p{};
  const size_t G = (size_t)(d->num_q_heads / d->num_kv_heads);
  const size_t slots = 2 * (size_t)ranges * G;
  p.ranges = ranges;
  p.ctrl_off = 0;
  p.layout_off = 256;
  p.ml_off = align256(p.layout_off + sizeof(int32_t) * 2 * (size_t)d->batch);
  p.o_off = align256(p.ml_off + sizeof(float2) * slots);
  p.total = align256(p.o_off + sizeof(float) * slots * d->head_dim);
  return p;
}

// The plan with the most ranges that fits in `bytes` (0 ranges if not even one fits).
WorkspacePlan fit_workspace(const pkv_dims* d, size_t bytes) {
  const WorkspacePlan base = plan_workspace(d, 0);
  const size_t G = (size_t)(d->num_q_heads / d->num_kv_heads);
  const size_t per_range = 2 * G * (sizeof(float2) + sizeof(float) * d->head_dim);
  // an upper estimate (alignment padding ignored), then down to the largest plan that fits
  long long r = bytes > base.total ? (long long)((bytes - base.total) / per_range) : 0;
  WorkspacePlan p = plan_workspace(d, r);
  while (r > 0 && p.total > bytes) p = plan_workspace(d, --r);
  return p;
}

namespace {

}  // namespace

int decode_common(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, const int32_t* kept,
                  const int32_t* kept_lens, int32_t max_kept, float scale, int32_t window,
                  void* workspace, size_t workspace_bytes, const pkv_dims* dims, int32_t* err,
                  void* stream, bool sparse, const void* k_new, const void* v_new,
                  const ScoreOutputs* score_out, const Q8Scales* q8, uint32_t flags) {
  int st = check_dims(dims, true);
  if (st != PKV_OK) return st;
  if (dims->batch > kMaxBatch) return PKV_ERR_DIMS;
  if ((flags & ~(uint32_t)PKV_DECODE_INPUTS_READY) != 0) return PKV_ERR_ARGUMENT;
  if (dims->batch == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return (!workspace) ? PKV_ERR_WORKSPACE : PKV_ERR_NULL_POINTER;
  if (sparse && (!kept || !kept_lens)) return PKV_ERR_NULL_POINTER;
  if (sparse && max_kept <= 0) return PKV_ERR_ARGUMENT;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace))
    return PKV_ERR_ALIGNMENT;
  const int group = dims->num_q_heads / dims->num_kv_heads;
  if (q8 != nullptr) {
    if (sparse && k_new != nullptr) return PKV_ERR_ARGUMENT;
    if (!q8->k_scale || !q8->v_scale) return PKV_ERR_NULL_POINTER;
    if (!aligned16(q8->k_scale) || !aligned16(q8->v_scale)) return PKV_ERR_ALIGNMENT;
  }
  if (score_out != nullptr) {
    if (sparse) return PKV_ERR_ARGUMENT;
    if (!score_out->lse || !score_out->scores || !score_out->logits) return PKV_ERR_NULL_POINTER;
    if (score_out->stride <= 0) return PKV_ERR_DIMS;
    if ((reinterpret_cast<uintptr_t>(score_out->lse) | reinterpret_cast<uintptr_t>(score_out->scores) |
         reinterpret_cast<uintptr_t>(score_out->logits)) & 3u)
      return PKV_ERR_ALIGNMENT;
  }
  const DecodeKernel k = decode_kernel(dims->head_dim, group, sparse, score_out != nullptr, q8 != nullptr);
  if (k.split == nullptr) return PKV_ERR_GQA;
  const int max_units = sparse ? (max_kept + 15) / 16 : dims->max_blocks_per_seq;
  // the flattened unit count and the pool's row count (a TMA coordinate) must fit int32
  if ((long long)dims->batch * dims->num_kv_heads * (long long)(max_units + 1) >= (1ll << 30))
    return PKV_ERR_DIMS;
  const long long pool_rows = (long long)dims->num_blocks * dims->num_kv_heads * PKV_BLOCK_SIZE;
  if (pool_rows >= (1ll << 31)) return PKV_ERR_DIMS;
  // partial slots for at least the static ranges of the largest grid
  const WorkspacePlan plan = fit_workspace(dims, workspace_bytes);
  if (plan.ranges < kMaxWorkers) return PKV_ERR_WORKSPACE;
  const DeviceInfo* info = device_info(&st);
  if (!info) return st;
  const size_t smem = decode_smem_bytes(dims->head_dim, sparse, dims->batch);
  const int mode = sparse ? (q8 ? 5 : 1) : (q8 ? (score_out ? 4 : 3) : (score_out ? 2 : 0));
  if (smem > info->max_dyn_smem[head_dim_index(dims->head_dim)][mode])
    return PKV_ERR_DIMS;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.split, kDecodeWarps * 32, smem);
  if (e != cudaSuccess) return cuda_status(e);
  if (per_sm < 1) return PKV_ERR_DIMS;

  DecodeArgs a{};
  if (q8 != nullptr) {  // the gather form copies rows one by one: no tensor maps
    if (!sparse) {
      st = encode_pool_map_q8(&a.tmap_k, k_cache, pool_rows, dims->head_dim);
      if (st == PKV_OK) st = encode_pool_map_q8(&a.tmap_v, v_cache, pool_rows, dims->head_dim);
      if (st != PKV_OK) return st;
    }
    a.k_scale = q8->k_scale;
    a.v_scale = q8->v_scale;
  } else if (!sparse) {
    st = encode_pool_map(&a.tmap_k, k_cache, pool_rows, dims->head_dim);
    if (st == PKV_OK) st = encode_pool_map(&a.tmap_v, v_cache, pool_rows, dims->head_dim);
    if (st != PKV_OK) return st;
  }
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.kept = kept;
  a.kept_lens = kept_lens;
  if (k_new != nullptr) {
    a.k_new = static_cast<const __nv_bfloat16*>(k_new);
    a.v_new = static_cast<const __nv_bfloat16*>(v_new);
    a.k_pool_out = static_cast<__nv_bfloat16*>(const_cast<void*>(k_cache));  // INT8: the code pools
    a.v_pool_out = static_cast<__nv_bfloat16*>(const_cast<void*>(v_cache));
    if (q8 != nullptr) {
      a.k_scale_out = const_cast<float*>(q8->k_scale);
      a.v_scale_out = const_cast<float*>(q8->v_scale);
    }
  }
  a.out = static_cast<__nv_bfloat16*>(out);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.ctrl = reinterpret_cast<uint32_t*>(ws + plan.ctrl_off);
  a.layout = reinterpret_cast<int32_t*>(ws + plan.layout_off);
  a.part_ml = reinterpret_cast<float2*>(ws + plan.ml_off);
  a.part_o = reinterpret_cast<float*>(ws + plan.o_off);
  if (score_out != nullptr) {
    a.logits = score_out->logits;
    a.lse = score_out->lse;
    a.scores = score_out->scores;
    a.score_stride = score_out->stride;
  }
  a.err = err;
  a.B = dims->batch;
  a.Hq = dims->num_q_heads;
  a.Hkv = dims->num_kv_heads;
  a.NB = dims->num_blocks;
  a.MB = dims->max_blocks_per_seq;
  a.max_kept = sparse ? max_kept : 0;
  a.window = sparse ? 0 : window;
  const int grid = std::min(info->sm_count * per_sm, kMaxWorkers / kDecodeWarps);
  const long long workers = (long long)grid * kDecodeWarps;
  a.workers = (int)workers;
  const int ring = (sparse && dims->head_dim == 128) ? PKV_RING_SPARSE_D128
                   : q8 != nullptr ? (dims->head_dim == 128 ? PKV_RING_Q8_D128 : PKV_RING_Q8_D64)
                                   : (dims->head_dim == 128 ? PKV_RING_D128 : PKV_RING_D64);
  // Partition settings by form (kernels.h has the measurements): the bf16 decode and its
  // score-emitting variant share one set, so their outputs agree bit for bit; the dense INT8
  // decode (issue-bound) and the gather form have their own.
  const bool dense_q8 = !sparse && q8 != nullptr;
  a.min_units = std::max(sparse ? PKV_MIN_UNITS_SPARSE : dense_q8 ? PKV_MIN_UNITS_Q8 : PKV_MIN_UNITS, 1);
  const int busy_pct = sparse ? (q8 != nullptr ? PKV_MIN_BUSY_PCT_SPARSE_Q8 : PKV_MIN_BUSY_PCT_SPARSE)
                       : dense_q8 ? PKV_MIN_BUSY_PCT_Q8 : PKV_MIN_BUSY_PCT;
  a.min_busy_pct = std::min(std::max(busy_pct, 0), 100);
  a.tail_pct = std::min(std::max(sparse ? PKV_TAIL_PCT_SPARSE : dense_q8 ? PKV_TAIL_PCT_Q8 : PKV_TAIL_PCT, 0), 50);
  a.chunk_min = std::max(dense_q8 ? PKV_CHUNK_MIN_Q8 : PKV_CHUNK_MIN, ring);  // never ends inside the tile ring
  a.cpw_cap = (int)std::min<long long>(std::min(PKV_MAX_TAIL_CHUNKS, kMaxTailChunksLimit),
                                       plan.ranges / workers - 1);
  a.early = (flags & PKV_DECODE_INPUTS_READY) != 0 ? 1 : 0;
  // A flagged call is usually followed by another (consecutive layers of a step): its merge
  // lets that call's split kernel launch at once, so the next prologue and first tile copies
  // overlap this call's last split warps.  Measured on one box, 28 qwen-shaped layers in a
  // graph: flagged bf16 0.848 -> 0.824 ms; unflagged bf16 0.918 -> 0.928 ms and flagged INT8
  // 0.743 -> 0.760 ms (issue-bound: the early prologues take issue slots from the tail), so
  // those keep the trigger after the merge's wait.
  a.merge_trigger_early = (a.early != 0 && q8 == nullptr) ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.timeout_ns = kWaitTimeoutNs;
  const int wpr_log2 = merge_warps_log2(
      dims, max_units, workers, a.min_units, a.min_busy_pct, a.tail_pct, a.chunk_min, a.cpw_cap,
      (long long)info->sm_count * info->merge_ctas_per_sm[head_dim_index(dims->head_dim)] * kMergeWarps,
      dense_q8 ? PKV_MERGE_PARTIALS_PER_WARP_Q8 : PKV_MERGE_PARTIALS_PER_WARP);
  return cuda_status(launch_decode(k, a, grid, smem, wpr_log2, static_cast<cudaStream_t>(stream)));
}


}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                  const int64_t* slot_mapping, int64_t num_tokens, const pkv_dims* dims,
                  int32_t* error_word, void* stream) {
  int st = check_dims(dims, false);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_DIMS;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PKV_ERR_NULL_POINTER;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k) || !aligned16(v))
    return PKV_ERR_ALIGNMENT;
  if (!device_info(&st)) return st;
  return cuda_status(launch_kv_append(k_cache, v_cache, k, v, slot_mapping, num_tokens,
                                      dims->num_kv_heads, dims->head_dim, dims->num_blocks,
                                      error_word, static_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_workspace_bytes(const pkv_dims* dims) {
  if (check_dims(dims, true) != PKV_OK || dims->batch > kMaxBatch) return 0;
  if (dims->num_q_heads / dims->num_kv_heads > kMaxGroup) return 0;
  return plan_workspace(dims, (long long)kMaxWorkers * (1 + std::min(PKV_MAX_TAIL_CHUNKS, kMaxTailChunksLimit))).total;
}

int pkv_paged_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               float scale, int32_t window, void* workspace,
                               size_t workspace_bytes, const pkv_dims* dims, uint32_t flags,
                               int32_t* error_word,
                               void* stream) {
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       window, workspace, workspace_bytes, dims, error_word, stream, false, nullptr, nullptr,
                       nullptr, nullptr, flags);
}

int pkv_kv_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k,
                     const void* v, const int64_t* slot_mapping, int64_t num_tokens, const pkv_dims* dims,
                     int32_t* error_word, void* stream) {
  int st = check_dims(dims, false);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_DIMS;
  if (num_tokens == 0) return PKV_OK;
  if (!k_codes || !v_codes || !k_scales || !v_scales || !k || !v || !slot_mapping) return PKV_ERR_NULL_POINTER;
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales) ||
      !aligned16(k) || !aligned16(v))
    return PKV_ERR_ALIGNMENT;
  if (!device_info(&st)) return st;
  return cuda_status(launch_kv_append_q8(k_codes, v_codes, k_scales, v_scales, k, v, slot_mapping, num_tokens,
                                         dims->num_kv_heads, dims->head_dim, dims->num_blocks, error_word,
                                         static_cast<cudaStream_t>(stream)));
}

int pkv_paged_decode_attention_q8(void* out, const void* q, const void* k_codes, const void* v_codes,
                                  const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                  const int32_t* context_lens, float scale, int32_t window, void* workspace,
                                  size_t workspace_bytes, const pkv_dims* dims, uint32_t flags,
                                  int32_t* error_word,
                                  void* stream) {
  const Q8Scales q8{k_scales, v_scales};
  return decode_common(out, q, k_codes, v_codes, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       window, workspace, workspace_bytes, dims, error_word, stream, false, nullptr, nullptr,
                       nullptr, &q8, flags);
}

int pkv_paged_decode_attention_append_q8(void* out, const void* q, void* k_codes, void* v_codes, float* k_scales,
                                         float* v_scales, const void* k_new, const void* v_new,
                                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                                         int32_t window, void* workspace, size_t workspace_bytes,
                                         const pkv_dims* dims, uint32_t flags, int32_t* error_word,
                                         void* stream) {
  if (k_new == nullptr || v_new == nullptr) return PKV_ERR_NULL_POINTER;
  if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGNMENT;
  const Q8Scales q8{k_scales, v_scales};
  return decode_common(out, q, k_codes, v_codes, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       window, workspace, workspace_bytes, dims, error_word, stream, false, k_new, v_new,
                       nullptr, &q8, flags);
}

int pkv_prefill_window_scores(float* score_accum, int32_t score_stride, float* lse, int32_t lse_given,
                              const void* q_win, const void* k_cache, const int32_t* block_tables,
                              const int32_t* context_lens, int32_t alpha, float scale, const pkv_dims* dims,
                              int32_t* error_word, void* stream) {
  int st = check_dims(dims, true);
  if (st != PKV_OK) return st;
  if (dims->batch > kMaxBatch) return PKV_ERR_DIMS;
  const int group = dims->num_q_heads / dims->num_kv_heads;
  if (group > kMaxGroup) return PKV_ERR_GQA;
  if (alpha <= 0 || score_stride <= 0) return PKV_ERR_ARGUMENT;
  if ((long long)alpha * group > kPrefillMaxColumns || dims->max_blocks_per_seq > kPrefillMaxBlocks)
    return PKV_ERR_DIMS;
  if (dims->batch == 0) return PKV_OK;
  if (!score_accum || !lse || !q_win || !k_cache || !block_tables || !context_lens) return PKV_ERR_NULL_POINTER;
  if (!aligned16(q_win) || !aligned16(k_cache) ||
      ((reinterpret_cast<uintptr_t>(score_accum) | reinterpret_cast<uintptr_t>(lse)) & 3u))
    return PKV_ERR_ALIGNMENT;
  const long long pool_rows = (long long)dims->num_blocks * dims->num_kv_heads * PKV_BLOCK_SIZE;
  if (pool_rows >= (1ll << 31) || (long long)dims->batch * alpha >= (1ll << 31) ||
      (long long)dims->max_blocks_per_seq * PKV_BLOCK_SIZE >= (1ll << 30))
    return PKV_ERR_DIMS;
  if (!device_info(&st)) return st;
  PrefillArgs a{};
  const int chunk_rows = 64 / group;
  st = encode_pool_map(&a.tmap_k, k_cache, pool_rows, dims->head_dim);
  if (st == PKV_OK)
    st = encode_window_map(&a.tmap_q, q_win, (long long)dims->batch * alpha, dims->num_q_heads, dims->head_dim,
                           group, chunk_rows);
  if (st != PKV_OK) return st;
  a.q_win = static_cast<const __nv_bfloat16*>(q_win);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.lse = lse;
  a.scores = score_accum;
  a.err = error_word;
  a.score_stride = score_stride;
  a.B = dims->batch;
  a.Hq = dims->num_q_heads;
  a.Hkv = dims->num_kv_heads;
  a.NB = dims->num_blocks;
  a.MB = dims->max_blocks_per_seq;
  a.alpha = alpha;
  a.G = group;
  a.R = chunk_rows;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.timeout_ns = kWaitTimeoutNs;
  return cuda_status(launch_prefill(a, dims->head_dim, lse_given != 0, static_cast<cudaStream_t>(stream)));
}

int pkv_paged_decode_attention_append(void* out, const void* q, void* k_cache, void* v_cache,
                                      const void* k_new, const void* v_new,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      float scale, int32_t window, void* workspace,
                                      size_t workspace_bytes, const pkv_dims* dims,
                                      uint32_t flags, int32_t* error_word, void* stream) {
  if (k_new == nullptr || v_new == nullptr) return PKV_ERR_NULL_POINTER;
  if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGNMENT;
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       window, workspace, workspace_bytes, dims, error_word, stream, false, k_new, v_new,
                       nullptr, nullptr, flags);
}

int pkv_paged_decode_attention_scores(void* out, float* lse_out, float* score_accum, float* logits,
                                      int32_t score_stride, const void* q, void* k_cache,
                                      void* v_cache, const void* k_new, const void* v_new,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      float scale, int32_t window, void* workspace,
                                      size_t workspace_bytes, const pkv_dims* dims,
                                      uint32_t flags, int32_t* error_word, void* stream) {
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_NULL_POINTER;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_ALIGNMENT;
  const ScoreOutputs so{lse_out, score_accum, logits, score_stride};
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       window, workspace, workspace_bytes, dims, error_word, stream, false, k_new, v_new, &so,
                       nullptr, flags);
}

int pkv_paged_decode_attention_scores_q8(void* out, float* lse_out, float* score_accum, float* logits,
                                         int32_t score_stride, const void* q, const void* k_codes,
                                         const void* v_codes, const float* k_scales, const float* v_scales,
                                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                                         int32_t window, void* workspace, size_t workspace_bytes,
                                         const pkv_dims* dims, uint32_t flags, int32_t* error_word,
                                         void* stream) {
  const ScoreOutputs so{lse_out, score_accum, logits, score_stride};
  const Q8Scales q8{k_scales, v_scales};
  return decode_common(out, q, k_codes, v_codes, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       window, workspace, workspace_bytes, dims, error_word, stream, false, nullptr, nullptr,
                       &so, &q8, flags);
}

size_t pkv_sparse_decode_workspace_bytes(const pkv_dims* dims, int32_t max_kept) {
  if (max_kept <= 0) return 0;
  return pkv_decode_workspace_bytes(dims);
}

int pkv_sparse_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* kept_index_lists, const int32_t* kept_lens,
                                int32_t max_kept, float scale, void* workspace,
                                size_t workspace_bytes, const pkv_dims* dims, uint32_t flags,
                                int32_t* error_word,
                                void* stream) {
  return decode_common(out, q, k_cache, v_cache, block_tables, context_lens, kept_index_lists, kept_lens,
                       max_kept, scale, 0, workspace, workspace_bytes, dims, error_word, stream, true,
                       nullptr, nullptr, nullptr, nullptr, flags);
}

int pkv_sparse_decode_attention_q8(void* out, const void* q, const void* k_codes, const void* v_codes,
                                   const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                   const int32_t* context_lens, const int32_t* kept_index_lists,
                                   const int32_t* kept_lens, int32_t max_kept, float scale, void* workspace,
                                   size_t workspace_bytes, const pkv_dims* dims, uint32_t flags,
                                   int32_t* error_word, void* stream) {
  const Q8Scales q8{k_scales, v_scales};
  return decode_common(out, q, k_codes, v_codes, block_tables, context_lens, kept_index_lists, kept_lens,
                       max_kept, scale, 0, workspace, workspace_bytes, dims, error_word, stream, true,
                       nullptr, nullptr, nullptr, &q8, flags);
}

int pkv_kv_select_topk(int32_t* kept_out, int32_t* kept_lens_out, const float* score_accum,
                       int32_t score_stride, const int32_t* context_lens, int32_t n_sink,
                       int32_t n_recent, int32_t k_top, const pkv_dims* dims, uint32_t flags,
                       int32_t* error_word, void* stream) {
  if (dims == nullptr) return PKV_ERR_NULL_POINTER;
  if ((flags & ~(uint32_t)PKV_SELECT_INPUTS_READY) != 0) return PKV_ERR_ARGUMENT;
  if (dims->batch < 0 || dims->num_kv_heads <= 0) return PKV_ERR_DIMS;
  if (n_sink < 0 || n_recent < 0 || k_top < 0 || score_stride < 0 || score_stride > 262144)
    return PKV_ERR_ARGUMENT;
  if ((long long)n_sink + n_recent + k_top > (1ll << 30)) return PKV_ERR_ARGUMENT;
  if (dims->batch == 0) return PKV_OK;
  if (!kept_out || !kept_lens_out || !score_accum || !context_lens) return PKV_ERR_NULL_POINTER;
  int st;
  if (!device_info(&st)) return st;
  return cuda_status(launch_select_topk(kept_out, kept_lens_out, score_accum, score_stride,
                                        context_lens, dims->batch, dims->num_kv_heads, n_sink,
                                        n_recent, k_top, (flags & PKV_SELECT_INPUTS_READY) ? 1 : 0,
                                        error_word, static_cast<cudaStream_t>(stream)));
}

int pkv_kv_compact(void* dst_k_cache, void* dst_v_cache, const int32_t* dst_block_tables,
                   int32_t dst_num_blocks, int32_t dst_max_blocks_per_seq, const void* src_k_cache,
                   const void* src_v_cache, const int32_t* src_block_tables,
                   const int32_t* context_lens, const int32_t* kept_index_lists,
                   const int32_t* kept_lens, int32_t max_kept, const pkv_dims* src_dims,
                   uint32_t flags, int32_t* error_word, void* stream) {
  if ((flags & ~(uint32_t)PKV_COMPACT_INPUTS_READY) != 0) return PKV_ERR_ARGUMENT;
  int st = check_dims(src_dims, false);
  if (st != PKV_OK) return st;
  if (dst_num_blocks < 0 || dst_max_blocks_per_seq < 0 || max_kept < 0) return PKV_ERR_DIMS;
  if (src_dims->batch == 0 || max_kept == 0) return PKV_OK;
  if (!dst_k_cache || !dst_v_cache || !dst_block_tables || !src_k_cache || !src_v_cache ||
      !src_block_tables || !context_lens || !kept_index_lists || !kept_lens)
    return PKV_ERR_NULL_POINTER;
  if (!aligned16(dst_k_cache) || !aligned16(dst_v_cache) || !aligned16(src_k_cache) ||
      !aligned16(src_v_cache))
    return PKV_ERR_ALIGNMENT;
  if (!device_info(&st)) return st;
  return cuda_status(launch_kv_compact(dst_k_cache, dst_v_cache, dst_block_tables, dst_num_blocks,
                                       dst_max_blocks_per_seq, src_k_cache, src_v_cache,
                                       src_block_tables, context_lens, kept_index_lists, kept_lens,
                                       max_kept, src_dims->batch, src_dims->num_kv_heads,
                                       src_dims->head_dim, src_dims->num_blocks,
                                       src_dims->max_blocks_per_seq,
                                       (flags & PKV_COMPACT_INPUTS_READY) ? 1 : 0, error_word,
                                       static_cast<cudaStream_t>(stream)));
}

int pkv_kv_compact_q8(void* dst_k_codes, void* dst_v_codes, float* dst_k_scales, float* dst_v_scales,
                      const int32_t* dst_block_tables, int32_t dst_num_blocks, int32_t dst_max_blocks_per_seq,
                      const void* src_k_codes, const void* src_v_codes, const float* src_k_scales,
                      const float* src_v_scales, const int32_t* src_block_tables, const int32_t* context_lens,
                      const int32_t* kept_index_lists, const int32_t* kept_lens, int32_t max_kept,
                      const pkv_dims* src_dims, uint32_t flags, int32_t* error_word, void* stream) {
  if ((flags & ~(uint32_t)PKV_COMPACT_INPUTS_READY) != 0) return PKV_ERR_ARGUMENT;
  int st = check_dims(src_dims, false);
  if (st != PKV_OK) return st;
  if (dst_num_blocks < 0 || dst_max_blocks_per_seq < 0 || max_kept < 0) return PKV_ERR_DIMS;
  if (src_dims->batch == 0 || max_kept == 0) return PKV_OK;
  if (!dst_k_codes || !dst_v_codes || !dst_k_scales || !dst_v_scales || !dst_block_tables || !src_k_codes ||
      !src_v_codes || !src_k_scales || !src_v_scales || !src_block_tables || !context_lens || !kept_index_lists ||
      !kept_lens)
    return PKV_ERR_NULL_POINTER;
  if (!aligned16(dst_k_codes) || !aligned16(dst_v_codes) || !aligned16(src_k_codes) || !aligned16(src_v_codes) ||
      !aligned16(dst_k_scales) || !aligned16(dst_v_scales) || !aligned16(src_k_scales) || !aligned16(src_v_scales))
    return PKV_ERR_ALIGNMENT;
  if (!device_info(&st)) return st;
  return cuda_status(launch_kv_compact_q8(
      dst_k_codes, dst_v_codes, dst_k_scales, dst_v_scales, dst_block_tables, dst_num_blocks, dst_max_blocks_per_seq,
      src_k_codes, src_v_codes, src_k_scales, src_v_scales, src_block_tables, context_lens, kept_index_lists,
      kept_lens, max_kept, src_dims->batch, src_dims->num_kv_heads, src_dims->head_dim, src_dims->num_blocks,
      src_dims->max_blocks_per_seq, (flags & PKV_COMPACT_INPUTS_READY) ? 1 : 0, error_word,
      static_cast<cudaStream_t>(stream)));
}

int pkv_kv_rolling_admit(void* k_cache, void* v_cache, const int32_t* block_tables,
                         int32_t* slot_pos, float* slot_score, int32_t* kept_lens,
                         const int32_t* context_lens, const void* k_new, const void* v_new,
                         int32_t capacity, int32_t n_sink, int32_t n_recent, const pkv_dims* dims,
                         uint32_t flags, int32_t* error_word, void* stream) {
  if ((flags & ~(uint32_t)PKV_ADMIT_INPUTS_READY) != 0) return PKV_ERR_ARGUMENT;
  int st = check_dims(dims, false);
  if (st != PKV_OK) return st;
  if (capacity <= 0 || n_sink < 0 || n_recent < 0 || (long long)n_sink + n_recent > capacity)
    return PKV_ERR_ARGUMENT;
  if ((long long)capacity > (long long)dims->max_blocks_per_seq * PKV_BLOCK_SIZE) return PKV_ERR_DIMS;
  if (dims->batch == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_tables || !slot_pos || !slot_score || !kept_lens ||
      !context_lens || !k_new || !v_new)
    return PKV_ERR_NULL_POINTER;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return PKV_ERR_ALIGNMENT;
  if (!device_info(&st)) return st;
  return cuda_status(launch_kv_rolling_admit(
      k_cache, v_cache, block_tables, dims->num_blocks, dims->max_blocks_per_seq, slot_pos, slot_score,
      kept_lens, context_lens, k_new, v_new, dims->batch, dims->num_kv_heads, dims->head_dim, capacity,
      n_sink, n_recent, (flags & PKV_ADMIT_INPUTS_READY) ? 1 : 0, error_word, static_cast<cudaStream_t>(stream)));
}

int pkv_kv_rolling_admit_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                            const int32_t* block_tables, int32_t* slot_pos, float* slot_score, int32_t* kept_lens,
                            const int32_t* context_lens, const void* k_new, const void* v_new, int32_t capacity,
                            int32_t n_sink, int32_t n_recent, const pkv_dims* dims, uint32_t flags,
                            int32_t* error_word, void* stream) {
  if ((flags & ~(uint32_t)PKV_ADMIT_INPUTS_READY) != 0) return PKV_ERR_ARGUMENT;
  int st = check_dims(dims, false);
  if (st != PKV_OK) return st;
  if (capacity <= 0 || n_sink < 0 || n_recent < 0 || (long long)n_sink + n_recent > capacity)
    return PKV_ERR_ARGUMENT;
  if ((long long)capacity > (long long)dims->max_blocks_per_seq * PKV_BLOCK_SIZE) return PKV_ERR_DIMS;
  if (dims->batch == 0) return PKV_OK;
  if (!k_codes || !v_codes || !k_scales || !v_scales || !block_tables || !slot_pos || !slot_score || !kept_lens ||
      !context_lens || !k_new || !v_new)
    return PKV_ERR_NULL_POINTER;
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales) ||
      !aligned16(k_new) || !aligned16(v_new))
    return PKV_ERR_ALIGNMENT;
  if (!device_info(&st)) return st;
  return cuda_status(launch_kv_rolling_admit_q8(
      k_codes, v_codes, k_scales, v_scales, block_tables, dims->num_blocks, dims->max_blocks_per_seq, slot_pos,
      slot_score, kept_lens, context_lens, k_new, v_new, dims->batch, dims->num_kv_heads, dims->head_dim, capacity,
      n_sink, n_recent, (flags & PKV_ADMIT_INPUTS_READY) ? 1 : 0, error_word, static_cast<cudaStream_t>(stream)));
}

int pkv_device_alias(const void* host_ptr, void** device_ptr) {
  if (host_ptr == nullptr || device_ptr == nullptr) return PKV_ERR_NULL_POINTER;
  *device_ptr = nullptr;
  // pinned (page-locked) host memory only: a system whose GPU reaches pageable memory too (a
  // Grace-Blackwell node) would map that as well, but its pages may move or be swapped out
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, host_ptr) != cudaSuccess || at.type != cudaMemoryTypeHost) {
    (void)cudaGetLastError();  // a host error, not a sticky one
    return PKV_ERR_ARGUMENT;
  }
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0) != cudaSuccess || d == nullptr) {
    (void)cudaGetLastError();
    return PKV_ERR_ARGUMENT;
  }
  *device_ptr = d;
  return PKV_OK;
}

int pkv_read_error(int32_t* error_word, int32_t clear, void* stream) {
  if (error_word == nullptr) return PKV_ERR_NULL_POINTER;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t value = 0;
  cudaError_t e = cudaMemcpyAsync(&value, error_word, sizeof(value), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) {
    e = cudaMemsetAsync(error_word, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return -(PKV_ERR_CUDA_BASE + (int)e);
  return value;
}

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PKV_ERR_DIMS: return "invalid or unsupported size";
    case PKV_ERR_BLOCK_SIZE: return "block_size must be 16";
    case PKV_ERR_HEAD_DIM: return "head_dim must be 64 or 128";
    case PKV_ERR_GQA: return "num_q_heads must be a multiple of num_kv_heads with G = Hq/Hkv <= 8";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_ALIGNMENT: return "a tensor pointer is not 16-byte aligned";
    case PKV_ERR_ARGUMENT: return "invalid scalar argument";
    case PKV_ERR_NO_DEVICE: return "no CUDA device";
    default: break;
  }
  if (status >= PKV_ERR_CUDA_BASE) return cudaGetErrorString(static_cast<cudaError_t>(status - PKV_ERR_CUDA_BASE));
  return "unknown status";
}

const char* pkv_device_error_string(int code) {
  switch (code) {
    case PKV_DEV_OK: return "no device error";
    case PKV_DEV_BAD_BLOCK_ID: return "block table entry outside the pool";
    case PKV_DEV_BAD_SLOT: return "slot outside the pool";
    case PKV_DEV_BAD_KEPT_INDEX: return "kept index outside the context";
    case PKV_DEV_BAD_CONTEXT_LEN: return "context length outside [0, max_blocks_per_seq*16]";
    case PKV_DEV_WAIT_TIMEOUT: return "a bounded wait timed out";
    case PKV_DEV_BAD_SCORE: return "NaN score";
    case PKV_DEV_DIRTY_WORKSPACE: return "decode workspace counters were not zero (zero-fill it before first use)";
    case PKV_DEV_BAD_VALUE: return "non-finite K/V element given to the INT8 append (token skipped)";
    default: return "unknown device error";
  }
}

}  // extern "C"
