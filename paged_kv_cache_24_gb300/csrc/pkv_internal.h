// pkv_internal.h -- shared definitions between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pkv {

// Tokens per work unit: one 16-row MMA tile of the context.
constexpr int kUnitTokens = 16;
// Warps per decode CTA; each warp streams its own units through its own
// shared-memory ring, and the warps merge their softmax states at the end.
constexpr int kDecodeWarps = 4;
// Ring depth (units in flight per warp) by head_dim, for 16-bit pools.
constexpr int kStagesD128 = 3;
constexpr int kStagesD64 = 4;
constexpr int kStagesFp8 = 3;  // 8-bit pools: 4 KB of codes + 128 B of scales per unit
// Bounded mbarrier wait (polls); a TMA that has not landed by then is treated
// as an error (output NaN), never as a reason to spin forever.
constexpr uint32_t kWaitLimit = 1u << 20;

// First position a length-L context attends with window `window`
// (window <= 0: no window).
__host__ __device__ __forceinline__ int window_start(int L, int window) {
  if (window <= 0) return 0;
  int lo = L - window;
  return lo > 0 ? lo : 0;
}

// The 16-token units a length-L context attends, as a virtual sequence
// 0 .. n_units-1: first the units holding the attention sinks [0, sinks),
// then the units of the window [lo, L).  When the two meet, one range from
// unit 0 covers both (tokens in a gap between them are masked per token).
struct SeqUnits {
  int lo;        // window start
  int sinks;     // sink positions before the window: [0, sinks)
  int n_sink_u;  // virtual units 0 .. n_sink_u-1 are physical units 0 .. n_sink_u-1
  int win_u0;    // virtual unit n_sink_u + i is physical unit win_u0 + i
  int n_units;
};

__host__ __device__ __forceinline__ SeqUnits seq_units(int L, int window, int num_sinks) {
  SeqUnits r{0, 0, 0, 0, 0};
  if (L <= 0) return r;
  r.lo = window_start(L, window);
  r.sinks = (window > 0 && num_sinks > 0) ? (num_sinks < r.lo ? num_sinks : r.lo) : 0;
  r.n_sink_u = (r.sinks + kUnitTokens - 1) / kUnitTokens;
  r.win_u0 = r.lo / kUnitTokens;
  if (r.n_sink_u >= r.win_u0) r.n_sink_u = r.win_u0 = 0;
  r.n_units = r.n_sink_u + (L + kUnitTokens - 1) / kUnitTokens - r.win_u0;
  return r;
}

__host__ __device__ __forceinline__ int phys_unit(const SeqUnits& r, int v) {
  return v < r.n_sink_u ? v : r.win_u0 + (v - r.n_sink_u);
}

// Is position t (0 <= t) attended by a length-L context?
__host__ __device__ __forceinline__ bool attended(const SeqUnits& r, int L, int t) {
  return t < L && (t >= r.lo || t < r.sinks);
}

__host__ __device__ __forceinline__ int splits_for(int n_units, int units_per_split) {
  return (n_units + units_per_split - 1) / units_per_split;
}

// Launch `kernel` so that it may be scheduled while the previous kernel in
// the stream finishes (programmatic stream serialisation).  Every kernel of
// this library calls pdl_wait_prior() before it reads global memory, so the
// overlap only hides launch latency.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DecodeParams {
  const void* q;               // [B][Hq][D]
  void* out;                   // [B][Hq][D]
  const void* k_cache;         // fp32 path reads the pools directly
  const void* v_cache;
  const int32_t* block_tables; // [B][MB]
  const int32_t* context_lens; // [B]
  const void* k_new;           // fused append: [B][Hkv][D] new keys (nullptr: decode only)
  const void* v_new;           //               [B][Hkv][D] new values
  void* k_dst;                 //               pools the new token is written to
  void* v_dst;
  const float* k_scale;        // FP8 pools: [NB][Hkv][bs] row scales (stored = code * scale)
  const float* v_scale;
  float* part_o;               // [B][Hq][S][D]  unnormalised partial outputs
  float2* part_ml;             // [B][Hq][S]     (running max in log2 units, sum)
  int64_t num_blocks;
  int num_seqs, num_q_heads, num_kv_heads, group;  // group = Hq / Hkv
  int head_chunk;              // query heads per CTA (<= 8 * NT)
  int num_head_chunks;         // ceil(group / head_chunk)
  int max_blocks;              // MB
  int block_size;              // bs
  int window;
  int num_sinks;               // attention sinks kept besides the window
  float scale_log2;            // scale * log2(e)
  int units_per_split;
  int num_splits;              // grid.x
};

// Launchers (return cudaGetLastError of the launch).
cudaError_t launch_decode_16bit(int dtype, int head_dim, int ntiles, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const DecodeParams& p,
                                cudaStream_t stream);
// FP8 E4M3 pools (head_dim 128), fp16 q / out; kmap / vmap describe the code pools.
// 8-bit pools (E4M3 codes, or int8 codes when `int8`), head_dim 128.
cudaError_t launch_decode_q8(bool int8, int ntiles, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_append_q8(bool int8, int in_dtype, const void* k, const void* v,
                             const int64_t* slots, int64_t num_tokens, void* k_codes,
                             void* v_codes, float* k_scale, float* v_scale, int64_t num_blocks,
                             int num_kv_heads, int block_size, int head_dim,
                             cudaStream_t stream);
cudaError_t launch_decode_f32(int head_dim, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_combine(int dtype, int head_dim, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_append(int elem_bytes, const void* k, const void* v, const int64_t* slots,
                          int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                          int num_kv_heads, int block_size, int head_dim, cudaStream_t stream);
cudaError_t launch_slot_mapping(const int32_t* block_tables, int num_seqs, int max_blocks,
                                const int64_t* positions, int block_size, int64_t* slots,
                                cudaStream_t stream);

// Device address of the library-resident split-K scratch buffer
// (PKV_NOALLOC_SCRATCH_BYTES) on `device`, which must be current.
int noalloc_scratch(int device, void** addr);
// Forget the looked-up addresses (pkv_release_workspaces; after a device reset).
void noalloc_forget();

}  // namespace pkv
