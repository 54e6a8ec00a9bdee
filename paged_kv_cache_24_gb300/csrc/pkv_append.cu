// pkv_append.cu -- slot mapping and the slot-mapped K/V append.
//
// "Build a Paged KV Cache in Pure Python", Step 3 (PagedKVCache.append): the
// token at position pos is written to row pos % block_size of the sequence's
// (pos // block_size)-th block.  Here the write is a pure 16-byte vector copy
// per thread, so the cache holds exactly the bits it was given.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int num_seqs,
                                    int max_blocks, const int64_t* __restrict__ positions,
                                    int block_size, int64_t* __restrict__ slots) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= num_seqs) return;
  const int64_t pos = positions[b];
  int64_t slot = -1;
  if (pos >= 0 && pos < static_cast<int64_t>(max_blocks) * block_size) {
    const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + pos / block_size];
    if (blk >= 0) slot = static_cast<int64_t>(blk) * block_size + pos % block_size;
  }
  slots[b] = slot;
}

// One thread per 16-byte chunk of one (token, kv head) row; K and V together.
__global__ void append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                              const int64_t* __restrict__ slots, int64_t num_tokens,
                              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                              int64_t num_blocks, int num_kv_heads, int block_size,
                              int chunks_per_row) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  if (idx >= num_tokens * per_token) return;
  const int64_t tok = idx / per_token;
  const int rem = static_cast<int>(idx - tok * per_token);
  const int h = rem / chunks_per_row;
  const int c = rem - h * chunks_per_row;
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_blocks * block_size) return;
  const int64_t blk = slot / block_size;
  const int64_t row = slot - blk * block_size;
  const int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * chunks_per_row + c;
  const int64_t src = idx;  // == (tok * Hkv + h) * chunks_per_row + c
  const uint4 kk = __ldg(k + src);
  const uint4 vv = __ldg(v + src);
  k_cache[dst] = kk;
  v_cache[dst] = vv;
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t* block_tables, int num_seqs, int max_blocks,
                                const int64_t* positions, int block_size, int64_t* slots,
                                cudaStream_t stream) {
  if (num_seqs == 0) return cudaSuccess;
  const int threads = 128;
  const int blocks = (num_seqs + threads - 1) / threads;
  return launch_pdl(slot_mapping_kernel, dim3(blocks), dim3(threads), 0, stream, block_tables,
                    num_seqs, max_blocks, positions, block_size, slots);
}

cudaError_t launch_append(int elem_bytes, const void* k, const void* v, const int64_t* slots,
                          int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                          int num_kv_heads, int block_size, int head_dim, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int chunks_per_row = head_dim * elem_bytes / 16;
  const int64_t total = num_tokens * num_kv_heads * chunks_per_row;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
                    num_tokens, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                    num_blocks, num_kv_heads, block_size, chunks_per_row);
}

}  // namespace pkv
