// pkv_prefill.h -- launchers of the paged chunked prefill (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Keys per tile of the tensor-core prefill, and query rows per CTA.
constexpr int kPrefillTileKeys = 128;
constexpr int kPrefillRowsCta = 256;

// A CTA's rows are (token, GQA head) pairs of one kv head: the largest power
// of two (at most 16) dividing the group size G is the number of heads per
// token, 256 / that the tokens per CTA.
__host__ __device__ __forceinline__ int prefill_heads_log2(int group) {
  int lg = 0;
  while (lg < 4 && group % (2 << lg) == 0) ++lg;
  return lg;
}

#ifdef __CUDACC__
// Work item (sequence b, token chunk c) of the prefill: the chunk's tokens
// tile0 .. tile0 + tile_n - 1 sit at positions pos0 .. pos1.  Their keys come
// in two sections of 128-key tiles, each tile holding consecutive positions:
//   sinks   (window > 0, num_sinks > 0): units 0 .. sink_units-1, which hold
//           the sink positions before the first row's window start k_lo,
//           padded to sink_tiles whole tiles;
//   window  units win_u0 .. pos1 / 16 (n_win_units of them), win_u0 =
//           max(k_lo / 16, sink_units), so that no unit is in both.
// `empty`: the chunk has no token there; `len_ok` false: the sequence's
// lengths are inconsistent (its rows become NaN).
struct PrefillItem {
  int start, n, tile0, tile_n, pos0, pos1, k_lo;
  int sink_units, sink_tiles, win_u0, n_win_units;
  int n_units, n_tiles;  // virtual units (sink tiles' units + window units), key tiles
  bool empty, len_ok;
};

__device__ __forceinline__ PrefillItem prefill_item(const int32_t* cu_q, const int32_t* lens,
                                                    int b, int c, int tok_per_cta, int window,
                                                    int num_sinks, int max_blocks,
                                                    int block_size) {
  constexpr int kTU = kPrefillTileKeys / 16;  // units per tile
  PrefillItem it{};
  it.start = cu_q[b];
  it.n = cu_q[b + 1] - it.start;
  it.tile0 = c * tok_per_cta;
  it.empty = it.tile0 >= it.n;
  if (it.empty) return it;
  const int L = lens[b];
  it.tile_n = min(tok_per_cta, it.n - it.tile0);
  it.pos0 = L - it.n + it.tile0;
  it.pos1 = it.pos0 + it.tile_n - 1;
  it.len_ok = L >= it.n && it.pos0 >= 0 &&
              static_cast<int64_t>(L) <= static_cast<int64_t>(max_blocks) * block_size;
  it.k_lo = window > 0 ? max(0, it.pos0 - window + 1) : 0;
  if (!it.len_ok) return it;
  const int sink_keys = (window > 0 && num_sinks > 0) ? min(num_sinks, it.k_lo) : 0;
  it.sink_units = (sink_keys + 15) / 16;
  it.sink_tiles = (it.sink_units + kTU - 1) / kTU;
  it.win_u0 = max(it.k_lo / 16, it.sink_units);
  it.n_win_units = it.pos1 / 16 - it.win_u0 + 1;  // >= 0: sink_units <= pos1 / 16 + 1
  it.n_units = it.sink_tiles * kTU + it.n_win_units;
  it.n_tiles = (it.n_units + kTU - 1) / kTU;
  return it;
}
#endif

// Chunked prefill: the chunk's rows to their slots, then attention.  The
// append launch also orders the work items (sequence, token chunk) by their
// number of key tiles, longest first, into `order` (num_seqs * chunks per
// sequence entries, device memory), and the attention CTAs take the items in
// that order: the hardware starts CTAs in index order, so the long items
// start first and the short ones fill the end (longest-processing-time-first).
// bf16 caches: the V range scan.  Each (sequence, kv head) gets row_blocks
// partial ranges of scan_rows context rows each: scan_rows a multiple of 128,
// at least 128, chosen so that row_blocks stays at most kPrefillScanParts (the
// attention's warps read a pair's partials two per lane, and the partials of
// a large batch stay a small buffer).
constexpr int kPrefillScanParts = 64;
struct PrefillScan {
  int scan_rows, row_blocks;
};
inline PrefillScan prefill_scan_plan(int max_blocks, int block_size) {
  const int64_t rows = static_cast<int64_t>(max_blocks) * block_size;
  const int64_t per = (rows + kPrefillScanParts - 1) / kPrefillScanParts;
  const int64_t sr = per <= 128 ? 128 : (per + 127) / 128 * 128;
  const int64_t rb = (rows + sr - 1) / sr;
  return PrefillScan{static_cast<int>(sr), static_cast<int>(rb > 0 ? rb : 1)};
}

// bf16 caches: `vparts` (num_seqs * num_kv_heads * row_blocks (max, min)
// pairs, device memory) receives, from the append launch, the range of each
// (sequence, kv head)'s V magnitudes over its context, from which the
// attention scales V into fp16 exactly, or leaves the pair to its exact bf16
// launch; `mode` (one word per attention CTA) carries that choice from the
// attention's first launch to its second.
cudaError_t launch_prefill(int dtype, int head_dim, const void* q, const void* k, const void* v,
                           const int32_t* cu_q, int num_seqs, int num_q_heads, int max_chunk,
                           void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads,
                           int block_size, const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, int window, int num_sinks, float scale,
                           void* out, int32_t* order, uint2* vparts, uint32_t* mode,
                           const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream);

// CTAs of the attention launch: one per (work item, kv head, head chunk).
inline int64_t prefill_ctas(int num_seqs, int num_q_heads, int num_kv_heads, int max_chunk) {
  const int group = num_q_heads / num_kv_heads;
  const int lg = prefill_heads_log2(group);
  const int tok_per_cta = kPrefillRowsCta >> lg;
  const int64_t chunks = (max_chunk + tok_per_cta - 1) / tok_per_cta;
  return static_cast<int64_t>(num_seqs) * chunks * num_kv_heads * (group >> lg);
}

// Attention half of the chunked prefill on the tcgen05 tensor cores (the
// chunk's rows must already be in the pools).
cudaError_t launch_prefill_tc(int dtype, int head_dim, const void* q, const int32_t* cu_q,
                              int num_seqs, int num_q_heads, int max_chunk, int64_t num_blocks,
                              int num_kv_heads, int block_size, const int32_t* block_tables,
                              int max_blocks, const int32_t* context_lens, int window,
                              int num_sinks, float scale, void* out, const int32_t* order,
                              const uint2* vparts, int row_blocks, uint32_t* mode,
                              const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream);

}  // namespace pkv
