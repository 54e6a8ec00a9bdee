// pkv_prefill.cu -- paged chunked prefill.
//
// What is computed ("Building a Streaming Sliding-Window Attention Engine in
// Pure Python", Step 3, prefill_attention: the mask (i - j) < window and
// j <= i, softmax per query row): sequence b holds L_b tokens after a chunk of
// n_b new ones was appended at positions L_b - n_b .. L_b - 1; the query of
// the chunk token at position p attends positions j <= p (and p - j < window
// when window > 0) of the paged cache -- the cached prefix and the chunk.
//
// How: the chunk's K/V rows are first written to their slots (the kernel
// below), then the attention runs on the tcgen05 tensor cores
// (pkv_prefill_tc.cu).
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_prefill.h"

namespace pkv {
namespace {

// The chunk's K/V rows to their slots: token i of sequence b sits at position
// L_b - n_b + i.  One thread per 16-byte chunk of a (token, kv head) row.
__global__ void chunk_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                    const int32_t* __restrict__ cu_q,
                                    const int32_t* __restrict__ context_lens,
                                    const int32_t* __restrict__ block_tables, int max_blocks,
                                    int block_size, int64_t num_blocks, int num_kv_heads,
                                    int chunks_per_row, uint4* __restrict__ k_cache,
                                    uint4* __restrict__ v_cache) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const int b = blockIdx.y;
  const int start = cu_q[b];
  const int n = cu_q[b + 1] - start;
  const int64_t per_tok = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n * per_tok) return;
  const int i = static_cast<int>(idx / per_tok);
  const int rem = static_cast<int>(idx - i * per_tok);
  const int h = rem / chunks_per_row, c = rem - h * chunks_per_row;
  const int64_t p = static_cast<int64_t>(context_lens[b]) - n + i;
  if (p < 0 || p >= static_cast<int64_t>(max_blocks) * block_size) return;
  const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + p / block_size];
  if (blk < 0 || blk >= num_blocks) return;
  const int64_t dst = ((static_cast<int64_t>(blk) * num_kv_heads + h) * block_size +
                       p % block_size) * chunks_per_row + c;
  const int64_t src = (static_cast<int64_t>(start + i) * num_kv_heads + h) * chunks_per_row + c;
  k_cache[dst] = __ldg(k + src);
  v_cache[dst] = __ldg(v + src);
}

}  // namespace

cudaError_t launch_prefill(int dtype, int head_dim, const void* q, const void* k, const void* v,
                           const int32_t* cu_q, int num_seqs, int num_q_heads, int max_chunk,
                           void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads,
                           int block_size, const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, int window, float scale, void* out,
                           const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream) {
  if (num_seqs == 0 || max_chunk == 0) return cudaSuccess;
  // 1) the chunk's rows to their slots
  const int cpr = head_dim * 2 / 16;
  const int64_t per_seq = static_cast<int64_t>(max_chunk) * num_kv_heads * cpr;
  dim3 agrid(static_cast<unsigned>((per_seq + 255) / 256), num_seqs);
  cudaError_t e = launch_pdl(chunk_append_kernel, agrid, dim3(256), 0, stream,
                             static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_q,
                             context_lens, block_tables, max_blocks, block_size, num_blocks,
                             num_kv_heads, cpr, static_cast<uint4*>(k_cache),
                             static_cast<uint4*>(v_cache));
  if (e != cudaSuccess) return e;
  // 2) attention over prefix + chunk on the tensor cores
  return launch_prefill_tc(dtype, head_dim, q, cu_q, num_seqs, num_q_heads, max_chunk,
                           num_blocks, num_kv_heads, block_size, block_tables, max_blocks,
                           context_lens, window, scale, out, kmap, vmap, stream);
}

}  // namespace pkv
