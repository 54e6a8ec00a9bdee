// pkv_prefill.h -- launchers of the paged chunked prefill (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Chunked prefill: the chunk's rows to their slots, then attention.
cudaError_t launch_prefill(int dtype, int head_dim, const void* q, const void* k, const void* v,
                           const int32_t* cu_q, int num_seqs, int num_q_heads, int max_chunk,
                           void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads,
                           int block_size, const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, int window, float scale, void* out,
                           const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream);

// Attention half of the chunked prefill on the tcgen05 tensor cores (the
// chunk's rows must already be in the pools).
cudaError_t launch_prefill_tc(int dtype, int head_dim, const void* q, const int32_t* cu_q,
                              int num_seqs, int num_q_heads, int max_chunk, int64_t num_blocks,
                              int num_kv_heads, int block_size, const int32_t* block_tables,
                              int max_blocks, const int32_t* context_lens, int window,
                              float scale, void* out, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t stream);

}  // namespace pkv
