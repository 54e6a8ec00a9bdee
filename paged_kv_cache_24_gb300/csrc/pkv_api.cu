// pkv_api.cu -- the C ABI of libpkv (declared in include/pkv.h): argument
// checks, split planning, the per-(device, stream) split-K workspace, TMA
// descriptor encoding and kernel dispatch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"
#include "pkv_prefill.h"
#include "pkv_stage.h"

namespace {

using pkv::DecodeParams;

// Tokens per split a caller may ask for, at most.
constexpr int kMaxSplitTokens = 65536;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int elem_bytes(int dtype) {
  return dtype == PKV_FLOAT32 ? 4 : ((dtype == PKV_FP8_E4M3 || dtype == PKV_INT8) ? 1 : 2);
}

// Layout checks.  `for_decode` adds the tile constraints of the decode kernels.
int check_layout(const pkv_cache_layout* L, bool for_decode) {
  if (!L) return PKV_ERR_NULL;
  if (L->dtype < PKV_FLOAT32 || L->dtype > PKV_INT8) return PKV_ERR_DTYPE;
  if (L->num_blocks < 0 || L->num_kv_heads <= 0 || L->block_size <= 0 || L->head_dim <= 0)
    return PKV_ERR_SHAPE;
  if ((L->head_dim * elem_bytes(L->dtype)) % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (for_decode) {
    if (L->head_dim != 64 && L->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if ((L->dtype == PKV_FP8_E4M3 || L->dtype == PKV_INT8) && L->head_dim != 128)
      return PKV_ERR_UNSUPPORTED;
    if (L->block_size % pkv::kUnitTokens != 0 || L->block_size > 256) return PKV_ERR_UNSUPPORTED;
    // TMA row coordinates are 32-bit
    if (L->num_blocks * L->num_kv_heads * static_cast<int64_t>(L->block_size) > 0x7fffffffLL)
      return PKV_ERR_UNSUPPORTED;
  }
  return PKV_OK;
}

int to_status(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  if (e == cudaErrorMemoryAllocation) return PKV_ERR_NOMEM;
  return PKV_ERR_CUDA;
}

// ---- split-K workspace, one per (device, stream) ---------------------------

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  std::vector<void*> retired;  // outgrown buffers, kept until pkv_release_workspaces
};
std::mutex g_ws_mutex;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// The stream's workspace, grown to `need` bytes.  An outgrown buffer is not
// freed: work already queued (or captured into a CUDA graph) may still use
// it, so it is retired and released only by pkv_release_workspaces.
int get_workspace(int device, cudaStream_t stream, size_t need, void** out) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  Workspace& ws = g_ws[{device, stream}];
  if (ws.bytes < need) {
    size_t bytes = need < (size_t(1) << 20) ? (size_t(1) << 20) : need;
    void* fresh = nullptr;
    cudaError_t e = cudaMalloc(&fresh, bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();  // clear the allocation error so later calls are unaffected
      return PKV_ERR_NOMEM;
    }
    if (ws.ptr) ws.retired.push_back(ws.ptr);
    ws.ptr = fresh;
    ws.bytes = bytes;
  }
  *out = ws.ptr;
  return PKV_OK;
}

// ---- TMA descriptors --------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The pool viewed as a 2-D tensor [NB * Hkv * bs rows][D columns]; one box is
// 16 rows x 64 columns (128 bytes) with the 128-byte swizzle.
int encode_pool_map(CUtensorMap* map, const void* pool, const pkv_cache_layout* L) {
  auto fn = get_encode_fn();
  if (!fn) return PKV_ERR_CUDA;
  const cuuint64_t rows = static_cast<cuuint64_t>(L->num_blocks) * L->num_kv_heads * L->block_size;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(L->head_dim), rows > 0 ? rows : 1};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(L->head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pkv::kUnitTokens)};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapDataType dt =
      L->dtype == PKV_FLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (L->dtype == PKV_FP8_E4M3 || L->dtype == PKV_INT8) {
    // code pools: one 128-byte box row per token row (head_dim 128)
    dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    strides[0] = static_cast<cuuint64_t>(L->head_dim);
    box[0] = static_cast<cuuint32_t>(L->head_dim);
  }
  CUresult r = fn(map, dt, 2, const_cast<void*>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// The decode kernels' view of a pool.  16-bit pools with head_dim 128 are
// seen as a 3-D tensor [2 column halves][NB * Hkv * bs rows][64 columns] (the
// halves' stride, 128 bytes, is below the rows' 256), so that one box of
// 64 x 16 x 2 brings a unit's 16 rows in a single copy, in shared memory as
// two 16 x 64 swizzled tiles one after the other; other pools keep the 2-D
// view above.
int encode_decode_map(CUtensorMap* map, const void* pool, const pkv_cache_layout* L) {
  if (L->head_dim != 128 || (L->dtype != PKV_FLOAT16 && L->dtype != PKV_BFLOAT16))
    return encode_pool_map(map, pool, L);
  auto fn = get_encode_fn();
  if (!fn) return PKV_ERR_CUDA;
  const cuuint64_t rows = static_cast<cuuint64_t>(L->num_blocks) * L->num_kv_heads * L->block_size;
  cuuint64_t dims[3] = {64, rows > 0 ? rows : 1, 2};
  cuuint64_t strides[2] = {256, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(pkv::kUnitTokens), 2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      L->dtype == PKV_FLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(map, dt, 3, const_cast<void*>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// ---- planning -----------------------------------------------------------------

struct Plan {
  int head_chunk, num_head_chunks, ntiles;
  int units_per_split, num_splits;
};

int sm_count_of_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int make_plan(int num_seqs, int num_q_heads, const pkv_cache_layout* L, int max_blocks,
              int window, int num_sinks, int tokens_per_split, int num_sms, Plan* plan) {
  const int group = num_q_heads / L->num_kv_heads;
  const int cap = L->dtype == PKV_FLOAT32 ? 8 : 16;  // query heads per CTA
  plan->head_chunk = group < cap ? group : cap;
  plan->num_head_chunks = (group + plan->head_chunk - 1) / plan->head_chunk;
  plan->ntiles = plan->head_chunk <= 8 ? 1 : 2;
  if (static_cast<int64_t>(L->num_kv_heads) * plan->num_head_chunks > 65535) return PKV_ERR_UNSUPPORTED;

  const int64_t total_units =
      static_cast<int64_t>(max_blocks) * L->block_size / pkv::kUnitTokens;
  int64_t max_units = total_units;
  if (window > 0) {
    // a window spans at most (w-1)/16 + 2 units; sinks add theirs in front
    const int64_t sink_units =
        num_sinks > 0 ? (static_cast<int64_t>(num_sinks) + pkv::kUnitTokens - 1) / pkv::kUnitTokens
                      : 0;
    const int64_t wu = (static_cast<int64_t>(window) - 1) / pkv::kUnitTokens + 2 + sink_units;
    if (wu < max_units) max_units = wu;
  }
  // The library's own plan starts at 2048 tokens per split (32 units per
  // warp, one lane each); a caller may ask for up to kMaxSplitTokens.
  const int max_ups = 32 * pkv::kDecodeWarps;
  const int cap_ups = kMaxSplitTokens / pkv::kUnitTokens;
  int ups;
  if (tokens_per_split > 0) {
    if (tokens_per_split % pkv::kUnitTokens != 0) return PKV_ERR_SHAPE;
    ups = tokens_per_split / pkv::kUnitTokens;
    if (ups > cap_ups) return PKV_ERR_UNSUPPORTED;
  } else {
    if (num_sms <= 0) num_sms = 148;
    const int64_t sms = num_sms;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * L->num_kv_heads * plan->num_head_chunks;
    // 16-bit pools at head_dim 128 with at most 8 query heads per CTA have a
    // twelve-warp kernel for grids of at most one CTA per SM
    const bool wide_kernel = L->head_dim == 128 && plan->ntiles == 1 &&
                             (L->dtype == PKV_FLOAT16 || L->dtype == PKV_BFLOAT16);
    if (wide_kernel && pairs <= sms) {
      // Fewer items than SMs: split each item into as many pieces as fit one
      // wave of one CTA per SM.  Measured on 4096-token contexts (32 query /
      // 8 kv heads, fp16), 1 / 4 / 12 sequences: 20.3 / 24.4 / 40.7 µs,
      // against 23.0 / 35.3 / 70.1 with the 128-token splits of the rule
      // below and 26.7 / 26.7 / 40.7 with one split per item.
      const int64_t ns_target = sms / pairs;
      int64_t u = (max_units + ns_target - 1) / ns_target;
      if (u < 1) u = 1;
      if (u > cap_ups) u = cap_ups;
      ups = static_cast<int>(u);
    } else {
      // Long splits cost the least per byte (each CTA pays its pipeline fill
      // and merge once): start at 2048 tokens and halve (down to 128) only
      // while the grid would give the SMs fewer than 4 CTAs each.
      const int64_t target = sms * 4;
      ups = max_ups;
      while (ups > 8 && pairs * ((max_units + ups - 1) / ups) < target) ups /= 2;
      // One split per item, with no combine pass, when no item can exceed
      // 257 units (4096 tokens at any alignment) and the items either balance
      // the SMs on their own (32 or more per SM: a serving batch of 8192
      // items of up to 2080 tokens, 5 % less time than 2048-token splits) or
      // fill at least four fifths of them one item each.
      if (max_units > ups && max_units <= 2 * max_ups + 1 &&
          (pairs >= 32 * sms || (pairs <= sms && 5 * pairs >= 4 * sms)))
        ups = static_cast<int>(max_units);
    }
  }
  int64_t ns = (max_units + ups - 1) / ups;
  if (ns < 1) ns = 1;
  if (ns > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  plan->units_per_split = ups;
  plan->num_splits = static_cast<int>(ns);
  return PKV_OK;
}

int check_decode_args(const void* q, int32_t num_seqs, int32_t num_q_heads, const void* k_cache,
                      const void* v_cache, const pkv_cache_layout* layout,
                      const int32_t* block_tables, int32_t max_blocks,
                      const int32_t* context_lens, const void* out) {
  int rc = check_layout(layout, true);
  if (rc != PKV_OK) return rc;
  if (num_seqs < 0 || num_q_heads <= 0 || max_blocks < 0) return PKV_ERR_SHAPE;
  if (num_q_heads % layout->num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * layout->block_size > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned4(block_tables) || !aligned4(context_lens))
    return PKV_ERR_ALIGNMENT;
  return PKV_OK;
}

// pkv_decode_split, optionally with the fused append of each sequence's token
// at position context_lens[b] - 1 (k_new / v_new non-null).
int decode_impl(const void* q, const void* k_new, const void* v_new, int32_t num_seqs,
                int32_t num_q_heads, const void* k_cache, const void* v_cache,
                const pkv_cache_layout* layout, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t window,
                int32_t num_sinks, float scale, void* out, int32_t tokens_per_split,
                void* stream, const float* k_scale = nullptr, const float* v_scale = nullptr,
                bool fixed_scratch = false) {
  int rc = check_decode_args(q, num_seqs, num_q_heads, k_cache, v_cache, layout, block_tables,
                             max_blocks_per_seq, context_lens, out);
  if (rc != PKV_OK) return rc;
  if (tokens_per_split < 0 || tokens_per_split % pkv::kUnitTokens != 0) return PKV_ERR_SHAPE;
  if (num_sinks < 0) return PKV_ERR_SHAPE;
  if (tokens_per_split > kMaxSplitTokens) return PKV_ERR_UNSUPPORTED;
  const bool q8 = layout->dtype == PKV_FP8_E4M3 || layout->dtype == PKV_INT8;
  if (q8 && num_seqs > 0) {
    if (!k_scale || !v_scale) return PKV_ERR_NULL;
    if (!aligned16(k_scale) || !aligned16(v_scale)) return PKV_ERR_ALIGNMENT;
    if (k_new) return PKV_ERR_UNSUPPORTED;
  }
  if (num_seqs == 0) return PKV_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PKV_ERR_CUDA;
  Plan plan;
  rc = make_plan(num_seqs, num_q_heads, layout, max_blocks_per_seq, window, num_sinks,
                 tokens_per_split, sm_count_of_current_device(), &plan);
  if (rc != PKV_OK) return rc;

  DecodeParams p{};
  p.q = q;
  p.out = out;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_dst = const_cast<void*>(k_cache);
  p.v_dst = const_cast<void*>(v_cache);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.num_blocks = layout->num_blocks;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = layout->num_kv_heads;
  p.group = num_q_heads / layout->num_kv_heads;
  p.head_chunk = plan.head_chunk;
  p.num_head_chunks = plan.num_head_chunks;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = layout->block_size;
  p.window = window;
  p.num_sinks = num_sinks;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.units_per_split = plan.units_per_split;
  p.num_splits = plan.num_splits;

  if (plan.num_splits > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * plan.num_splits;
    const size_t o_bytes = rows * layout->head_dim * sizeof(float);
    const size_t need = o_bytes + rows * sizeof(float2);
    void* ws = nullptr;
    if (fixed_scratch) {
      // the buffer in the library image (pkv_noalloc.cu): no allocation
      if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_SCRATCH;
      rc = pkv::noalloc_scratch(device, &ws);
    } else {
      rc = get_workspace(device, st, need, &ws);
    }
    if (rc != PKV_OK) return rc;
    p.part_o = static_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + o_bytes);
  }

  cudaError_t e;
  if (layout->dtype == PKV_FLOAT32) {
    e = pkv::launch_decode_f32(layout->head_dim, p, st);
  } else {
    CUtensorMap kmap, vmap;
    rc = encode_decode_map(&kmap, k_cache, layout);
    if (rc != PKV_OK) return rc;
    rc = encode_decode_map(&vmap, v_cache, layout);
    if (rc != PKV_OK) return rc;
    e = q8 ? pkv::launch_decode_q8(layout->dtype == PKV_INT8, plan.ntiles, kmap, vmap, p, st)
            : pkv::launch_decode_16bit(layout->dtype, layout->head_dim, plan.ntiles, kmap, vmap,
                                       p, st);
  }
  if (e != cudaSuccess) return to_status(e);
  if (plan.num_splits > 1) {
    // 8-bit pools decode into fp16 outputs
    e = pkv::launch_combine(q8 ? PKV_FLOAT16 : layout->dtype, layout->head_dim, p, st);
    if (e != cudaSuccess) return to_status(e);
  }
  return PKV_OK;
}

}  // namespace



// Quantising append into an 8-bit pool (E4M3 or int8 codes).
static int append_q8(bool int8, const void* k, const void* v, int32_t in_dtype,
                     const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                     void* v_cache, float* k_scale, float* v_scale,
                     const pkv_cache_layout* layout, void* stream) {
  int rc = check_layout(layout, false);
  if (rc != PKV_OK) return rc;
  if (layout->dtype != (int8 ? PKV_INT8 : PKV_FP8_E4M3)) return PKV_ERR_DTYPE;
  if (in_dtype < PKV_FLOAT32 || in_dtype > PKV_BFLOAT16) return PKV_ERR_DTYPE;
  if (layout->head_dim != 64 && layout->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned4(k_scale) || !aligned4(v_scale) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_ALIGNMENT;
  return to_status(pkv::launch_append_q8(int8, in_dtype, k, v, slot_mapping, num_tokens, k_cache,
                                         v_cache, k_scale, v_scale, layout->num_blocks,
                                         layout->num_kv_heads, layout->block_size,
                                         layout->head_dim, static_cast<cudaStream_t>(stream)));
}


extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: negative or inconsistent sizes";
    case PKV_ERR_DTYPE: return "PKV_ERR_DTYPE: unknown dtype code";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: shape or size not supported";
    case PKV_ERR_ALIGNMENT: return "PKV_ERR_ALIGNMENT: data pointer not 16-byte aligned";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA call or kernel launch failed";
    case PKV_ERR_NOMEM: return "PKV_ERR_NOMEM: workspace allocation failed";
    case PKV_ERR_SCRATCH: return "PKV_ERR_SCRATCH: problem needs more than the fixed no-alloc scratch";
    case PKV_ERR_RANGE: return "PKV_ERR_RANGE: an index is out of range (pkv_validate_indices)";
    default: return "unknown pkv status";
  }
}

int pkv_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                     const int64_t* positions, int32_t block_size, int64_t* slot_mapping,
                     void* stream) {
  if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (!block_tables || !positions || !slot_mapping) return PKV_ERR_NULL;
  if (!aligned4(block_tables) || (reinterpret_cast<uintptr_t>(positions) & 7u) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_ALIGNMENT;
  return to_status(pkv::launch_slot_mapping(block_tables, num_seqs, max_blocks_per_seq, positions,
                                            block_size, slot_mapping,
                                            static_cast<cudaStream_t>(stream)));
}

// The address a kernel uses for p: p itself for device or managed memory, the
// device-side address of pinned host memory; nullptr when no kernel may touch p
// (pageable host memory, or no CUDA allocation at all).
static const void* device_side(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // not a CUDA pointer: clear the error
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

int pkv_device_address(const void* p, void** device_address) {
  if (!device_address) return PKV_ERR_NULL;
  *device_address = nullptr;
  if (!p) return PKV_ERR_NULL;
  const void* d = device_side(p);
  if (!d) return PKV_ERR_UNSUPPORTED;
  *device_address = const_cast<void*>(d);
  return PKV_OK;
}

int pkv_stage_copy(void* dst, const void* src, int64_t bytes, void* stream) {
  if (bytes < 0) return PKV_ERR_SHAPE;
  if (bytes == 0) return PKV_OK;
  if (!dst || !src) return PKV_ERR_NULL;
  if (!aligned16(dst) || !aligned16(src)) return PKV_ERR_ALIGNMENT;
  const void* d = device_side(dst);
  const void* s = device_side(src);
  if (!d || !s) return PKV_ERR_UNSUPPORTED;
  return to_status(pkv::launch_stage_copy(const_cast<void*>(d), s, bytes,
                                          sm_count_of_current_device(),
                                          static_cast<cudaStream_t>(stream)));
}

int pkv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
               void* k_cache, void* v_cache, const pkv_cache_layout* layout, void* stream) {
  int rc = check_layout(layout, false);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_ALIGNMENT;
  return to_status(pkv::launch_append(elem_bytes(layout->dtype), k, v, slot_mapping, num_tokens,
                                      k_cache, v_cache, layout->num_blocks, layout->num_kv_heads,
                                      layout->block_size, layout->head_dim,
                                      static_cast<cudaStream_t>(stream)));
}

int pkv_decode_plan(int32_t num_seqs, int32_t num_q_heads, const pkv_cache_layout* layout,
                    int32_t max_blocks_per_seq, int32_t window, int32_t num_sinks,
                    int32_t tokens_per_split, int32_t num_sms, int32_t* tokens_per_split_out,
                    int32_t* num_splits_out) {
  int rc = check_layout(layout, true);
  if (rc != PKV_OK) return rc;
  if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq < 0 ||
      num_q_heads % layout->num_kv_heads != 0)
    return PKV_ERR_SHAPE;
  if (num_sinks < 0) return PKV_ERR_SHAPE;
  Plan plan;
  rc = make_plan(num_seqs, num_q_heads, layout, max_blocks_per_seq, window, num_sinks,
                 tokens_per_split, num_sms > 0 ? num_sms : sm_count_of_current_device(), &plan);
  if (rc != PKV_OK) return rc;
  if (tokens_per_split_out) *tokens_per_split_out = plan.units_per_split * pkv::kUnitTokens;
  if (num_splits_out) *num_splits_out = plan.num_splits;
  return PKV_OK;
}

int pkv_decode_split(const void* q, int32_t num_seqs, int32_t num_q_heads,
                     const void* k_cache, const void* v_cache, const pkv_cache_layout* layout,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, int32_t window, float scale, void* out,
                     int32_t tokens_per_split, void* stream) {
  return decode_impl(q, nullptr, nullptr, num_seqs, num_q_heads, k_cache, v_cache, layout,
                     block_tables, max_blocks_per_seq, context_lens, window, 0, scale, out,
                     tokens_per_split, stream);
}

static int decode_options_impl(const void* q, int32_t num_seqs, int32_t num_q_heads,
                               void* k_cache, void* v_cache, const pkv_cache_layout* layout,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, float scale, void* out,
                               const pkv_decode_options* options, void* stream,
                               bool fixed_scratch) {
  if (!options) return PKV_ERR_NULL;
  if (num_seqs > 0 && (options->k_new != nullptr) != (options->v_new != nullptr))
    return PKV_ERR_NULL;
  if (num_seqs > 0 && options->k_new &&
      (!aligned16(options->k_new) || !aligned16(options->v_new)))
    return PKV_ERR_ALIGNMENT;
  return decode_impl(q, options->k_new, options->v_new, num_seqs, num_q_heads, k_cache, v_cache,
                     layout, block_tables, max_blocks_per_seq, context_lens, options->window,
                     options->num_sinks, scale, out, options->tokens_per_split, stream,
                     options->k_scale, options->v_scale, fixed_scratch);
}

int pkv_decode_ex(const void* q, int32_t num_seqs, int32_t num_q_heads, void* k_cache,
                  void* v_cache, const pkv_cache_layout* layout, const int32_t* block_tables,
                  int32_t max_blocks_per_seq, const int32_t* context_lens, float scale, void* out,
                  const pkv_decode_options* options, void* stream) {
  return decode_options_impl(q, num_seqs, num_q_heads, k_cache, v_cache, layout, block_tables,
                             max_blocks_per_seq, context_lens, scale, out, options, stream,
                             false);
}

int pkv_decode_noalloc_ex(const void* q, int32_t num_seqs, int32_t num_q_heads, void* k_cache,
                          void* v_cache, const pkv_cache_layout* layout,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, float scale, void* out,
                          const pkv_decode_options* options, void* stream) {
  return decode_options_impl(q, num_seqs, num_q_heads, k_cache, v_cache, layout, block_tables,
                             max_blocks_per_seq, context_lens, scale, out, options, stream,
                             true);
}

int pkv_decode_noalloc(const void* q, int32_t num_seqs, int32_t num_q_heads,
                       const void* k_cache, const void* v_cache, const pkv_cache_layout* layout,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t window, float scale, void* out,
                       void* stream) {
  // 8-bit pools need row scales, which this form does not take
  if (layout && (layout->dtype == PKV_FP8_E4M3 || layout->dtype == PKV_INT8))
    return PKV_ERR_UNSUPPORTED;
  return decode_impl(q, nullptr, nullptr, num_seqs, num_q_heads, k_cache, v_cache, layout,
                     block_tables, max_blocks_per_seq, context_lens, window, 0, scale, out, 0,
                     stream, nullptr, nullptr, true);
}

int pkv_prefill(const void* q, const void* k, const void* v, const int32_t* cu_q,
                int32_t num_seqs, int32_t num_q_heads, int32_t max_chunk, void* k_cache,
                void* v_cache, const pkv_cache_layout* layout, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t window,
                int32_t num_sinks, float scale, void* out, void* stream) {
  int rc = check_layout(layout, true);
  if (rc != PKV_OK) return rc;
  if (layout->dtype != PKV_FLOAT16 && layout->dtype != PKV_BFLOAT16) return PKV_ERR_UNSUPPORTED;
  if (num_seqs < 0 || num_q_heads <= 0 || max_chunk < 0 || max_blocks_per_seq < 0 ||
      num_sinks < 0 || num_q_heads % layout->num_kv_heads != 0)
    return PKV_ERR_SHAPE;
  if (num_seqs > 65534) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * layout->block_size > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;  // positions are 32-bit
  if (num_seqs == 0 || max_chunk == 0) return PKV_OK;
  // work items (sequence, token chunk) and their CTAs (one per kv head and head chunk)
  const int group = num_q_heads / layout->num_kv_heads;
  const int heads_log2 = pkv::prefill_heads_log2(group);
  const int tok_per_cta = pkv::kPrefillRowsCta >> heads_log2;
  const int64_t items = static_cast<int64_t>(num_seqs) * ((max_chunk + tok_per_cta - 1) / tok_per_cta);
  if (items * layout->num_kv_heads * (group >> heads_log2) > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  if (!q || !k || !v || !cu_q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || !aligned4(cu_q) || !aligned4(block_tables) ||
      !aligned4(context_lens))
    return PKV_ERR_ALIGNMENT;
  CUtensorMap kmap, vmap;
  rc = encode_pool_map(&kmap, k_cache, layout);
  if (rc != PKV_OK) return rc;
  rc = encode_decode_map(&vmap, v_cache, layout);  // 3-D for head_dim 128: one copy per V unit
  if (rc != PKV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PKV_ERR_CUDA;
  // written and read on this stream: the items' order; bf16 caches: each
  // (sequence, kv head)'s partial V ranges and each attention CTA's mode word
  auto align16 = [](size_t x) { return (x + 15) & ~size_t(15); };
  const size_t order_bytes = align16(static_cast<size_t>(items) * sizeof(int32_t));
  const pkv::PrefillScan scan = pkv::prefill_scan_plan(max_blocks_per_seq, layout->block_size);
  const bool bf16 = layout->dtype == PKV_BFLOAT16;
  const size_t parts_bytes =
      bf16 ? align16(static_cast<size_t>(num_seqs) * layout->num_kv_heads * scan.row_blocks * 8)
           : 0;
  const size_t mode_bytes =
      bf16 ? static_cast<size_t>(pkv::prefill_ctas(num_seqs, num_q_heads, layout->num_kv_heads,
                                                   max_chunk)) * sizeof(uint32_t)
           : 0;
  void* ws = nullptr;
  rc = get_workspace(device, st, order_bytes + parts_bytes + mode_bytes, &ws);
  if (rc != PKV_OK) return rc;
  char* wsb = static_cast<char*>(ws);
  return to_status(pkv::launch_prefill(
      layout->dtype, layout->head_dim, q, k, v, cu_q, num_seqs, num_q_heads, max_chunk, k_cache,
      v_cache, layout->num_blocks, layout->num_kv_heads, layout->block_size, block_tables,
      max_blocks_per_seq, context_lens, window, num_sinks, scale, out,
      reinterpret_cast<int32_t*>(wsb), bf16 ? reinterpret_cast<uint2*>(wsb + order_bytes) : nullptr,
      bf16 ? reinterpret_cast<uint32_t*>(wsb + order_bytes + parts_bytes) : nullptr, kmap, vmap,
      st));
}

int pkv_append_fp8(const void* k, const void* v, int32_t in_dtype, const int64_t* slot_mapping,
                   int64_t num_tokens, void* k_cache, void* v_cache, float* k_scale,
                   float* v_scale, const pkv_cache_layout* layout, void* stream) {
  return append_q8(false, k, v, in_dtype, slot_mapping, num_tokens, k_cache, v_cache, k_scale,
                   v_scale, layout, stream);
}

int pkv_append_int8(const void* k, const void* v, int32_t in_dtype, const int64_t* slot_mapping,
                    int64_t num_tokens, void* k_cache, void* v_cache, float* k_scale,
                    float* v_scale, const pkv_cache_layout* layout, void* stream) {
  return append_q8(true, k, v, in_dtype, slot_mapping, num_tokens, k_cache, v_cache, k_scale,
                   v_scale, layout, stream);
}

int pkv_append_decode(const void* q, const void* k_new, const void* v_new, int32_t num_seqs,
                      int32_t num_q_heads, void* k_cache, void* v_cache,
                      const pkv_cache_layout* layout, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t window,
                      float scale, void* out, int32_t tokens_per_split, void* stream) {
  if (num_seqs > 0) {
    if (!k_new || !v_new) return PKV_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGNMENT;
  }
  return decode_impl(q, k_new, v_new, num_seqs, num_q_heads, k_cache, v_cache, layout,
                     block_tables, max_blocks_per_seq, context_lens, window, 0, scale, out,
                     tokens_per_split, stream);
}

int pkv_decode(const void* q, int32_t num_seqs, int32_t num_q_heads, const void* k_cache,
               const void* v_cache, const pkv_cache_layout* layout, const int32_t* block_tables,
               int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t window,
               float scale, void* out, void* stream) {
  return pkv_decode_split(q, num_seqs, num_q_heads, k_cache, v_cache, layout, block_tables,
                          max_blocks_per_seq, context_lens, window, scale, out, 0, stream);
}

int pkv_validate_indices(const int32_t* block_tables, int32_t num_seqs,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         const int64_t* slot_mapping, int64_t num_slots, int64_t num_blocks,
                         int32_t block_size, void* stream, pkv_index_error* error) {
  if (error) *error = pkv_index_error{0, 0, 0, 0};
  if (num_seqs < 0 || max_blocks_per_seq < 0 || num_slots < 0 || num_blocks < 0 ||
      block_size < 1)
    return PKV_ERR_SHAPE;
  if ((num_seqs > 0 && (!block_tables || !context_lens)) || (num_slots > 0 && !slot_mapping))
    return PKV_ERR_NULL;
  auto fail = [&](int what, int64_t row, int64_t col, int64_t value) {
    if (error) *error = pkv_index_error{what, row, col, value};
    return PKV_ERR_RANGE;
  };
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t n_table = static_cast<size_t>(num_seqs) * static_cast<size_t>(max_blocks_per_seq);
  std::vector<int32_t> lens(static_cast<size_t>(num_seqs)), table(n_table);
  std::vector<int64_t> slots(static_cast<size_t>(num_slots));
  auto fetch = [&](void* dst, const void* src, size_t bytes) {
    return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, st) == cudaSuccess;
  };
  if (!fetch(lens.data(), context_lens, lens.size() * sizeof(int32_t)) ||
      !fetch(table.data(), block_tables, table.size() * sizeof(int32_t)) ||
      !fetch(slots.data(), slot_mapping, slots.size() * sizeof(int64_t)) ||
      ((num_seqs > 0 || num_slots > 0) && cudaStreamSynchronize(st) != cudaSuccess)) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  const int64_t max_len = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  for (int32_t b = 0; b < num_seqs; ++b)
    if (lens[b] < 0 || lens[b] > max_len) return fail(1, b, 0, lens[b]);
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int64_t used = (static_cast<int64_t>(lens[b]) + block_size - 1) / block_size;
    for (int64_t j = 0; j < used; ++j) {
      const int32_t e = table[static_cast<size_t>(b) * max_blocks_per_seq + j];
      if (e < 0 || e >= num_blocks) return fail(2, b, j, e);
    }
  }
  const int64_t pool_slots = num_blocks * block_size;
  std::vector<std::pair<int64_t, int64_t>> taken;  // (slot, token)
  taken.reserve(slots.size());
  for (int64_t i = 0; i < num_slots; ++i) {
    if (slots[i] >= pool_slots) return fail(3, i, 0, slots[i]);
    if (slots[i] >= 0) taken.emplace_back(slots[i], i);
  }
  std::sort(taken.begin(), taken.end());
  // the earliest token whose slot an earlier token already holds: in each run
  // of equal slots (tokens ascending) the run's second token
  int64_t row = -1, col = -1, value = 0;
  for (size_t k = 1; k < taken.size(); ++k) {
    const bool second = taken[k].first == taken[k - 1].first &&
                        (k == 1 || taken[k - 1].first != taken[k - 2].first);
    if (second && (row < 0 || taken[k].second < row)) {
      row = taken[k].second;
      col = taken[k - 1].second;
      value = taken[k].first;
    }
  }
  if (row >= 0) return fail(4, row, col, value);
  return PKV_OK;
}

int pkv_release_workspaces(void) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  int rc = PKV_OK;
  if (!g_ws.empty() && cudaDeviceSynchronize() != cudaSuccess) rc = PKV_ERR_CUDA;
  int prev = 0;
  cudaGetDevice(&prev);
  for (auto& kv : g_ws) {
    cudaSetDevice(kv.first.first);
    if (kv.second.ptr) cudaFree(kv.second.ptr);
    for (void* r : kv.second.retired) cudaFree(r);
  }
  cudaSetDevice(prev);
  g_ws.clear();
  pkv::noalloc_forget();
  return rc;
}

}  // extern "C"
