// pkv_prefill.cu -- paged chunked prefill.
//
// What is computed ("Building a Streaming Sliding-Window Attention Engine in
// Pure Python", Step 3, prefill_attention: the mask (i - j) < window and
// j <= i, softmax per query row): sequence b holds L_b tokens after a chunk of
// n_b new ones was appended at positions L_b - n_b .. L_b - 1; the query of
// the chunk token at position p attends positions j <= p (and p - j < window
// when window > 0) of the paged cache -- the cached prefix and the chunk.
// With a window, the first num_sinks positions stay attended as well
// ("Building a Streaming Sliding-Window Attention Engine in Pure Python",
// Extending: the StreamingLLM attention-sink item).
//
// How: the chunk's K/V rows are first written to their slots (the kernel
// below, whose extra block also orders the attention's work items), then the
// attention runs on the tcgen05 tensor cores (pkv_prefill_tc.cu).
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_prefill.h"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kAppendVec = 4;  // 16-byte chunks per thread (a row has 8 or 16)
constexpr int kPlanBins = 1024;  // work sizes 0 .. 1023 key tiles (larger ones share the top bin)
constexpr int kPlanCache = 4;    // planner items per thread sized once

struct PlanArgs {
  int32_t* order;
  int chunks_per_seq, tok_per_cta, window, num_sinks;
};

// Work items (sequence b, token chunk c), item id b * chunks_per_seq + c, in
// descending order of their key tiles: a counting sort over the work sizes in
// one block (histogram, exclusive scan, scatter).  Items of equal size come
// in any order; each item's result does not depend on when it runs.
__device__ void plan_items(const int32_t* __restrict__ cu_q,
                           const int32_t* __restrict__ context_lens, int num_seqs,
                           int max_blocks, int block_size, const PlanArgs& pa) {
  static_assert(kPlanBins == 4 * kAppendThreads, "four bins per thread");
  __shared__ __align__(16) int bins[kPlanBins];
  __shared__ int warp_sum[kAppendThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  reinterpret_cast<int4*>(bins)[tid] = make_int4(0, 0, 0, 0);
  __syncthreads();
  const int64_t n_items = static_cast<int64_t>(num_seqs) * pa.chunks_per_seq;
  auto bin_of = [&](int64_t i) {
    const int b = static_cast<int>(i / pa.chunks_per_seq);
    const int c = static_cast<int>(i - static_cast<int64_t>(b) * pa.chunks_per_seq);
    const PrefillItem it = prefill_item(cu_q, context_lens, b, c, pa.tok_per_cta, pa.window,
                                        pa.num_sinks, max_blocks, block_size);
    const int w = it.empty ? 0 : min(it.n_tiles, kPlanBins - 1);
    return kPlanBins - 1 - w;  // the largest work first
  };
  // the first kPlanCache items of each thread keep their bin in registers (their
  // reads all go out before the first one is used); any further ones are
  // sized twice
  int cached[kPlanCache];
#pragma unroll
  for (int r = 0; r < kPlanCache; ++r) {
    const int64_t i = tid + static_cast<int64_t>(r) * kAppendThreads;
    cached[r] = i < n_items ? bin_of(i) : 0;
  }
#pragma unroll
  for (int r = 0; r < kPlanCache; ++r)
    if (tid + static_cast<int64_t>(r) * kAppendThreads < n_items) atomicAdd(&bins[cached[r]], 1);
  for (int64_t i = tid + static_cast<int64_t>(kPlanCache) * kAppendThreads; i < n_items;
       i += kAppendThreads)
    atomicAdd(&bins[bin_of(i)], 1);
  __syncthreads();
  // exclusive scan: thread t owns bins 4t .. 4t + 3 (one 16-byte access each way)
  const int4 c4 = reinterpret_cast<const int4*>(bins)[tid];
  const int local = c4.x + c4.y + c4.z + c4.w;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += warp_sum[w];
  int4 first;
  first.x = run;
  first.y = first.x + c4.x;
  first.z = first.y + c4.y;
  first.w = first.z + c4.z;
  reinterpret_cast<int4*>(bins)[tid] = first;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kPlanCache; ++r) {
    const int64_t i = tid + static_cast<int64_t>(r) * kAppendThreads;
    if (i < n_items) pa.order[atomicAdd(&bins[cached[r]], 1)] = static_cast<int32_t>(i);
  }
  for (int64_t i = tid + static_cast<int64_t>(kPlanCache) * kAppendThreads; i < n_items;
       i += kAppendThreads)
    pa.order[atomicAdd(&bins[bin_of(i)], 1)] = static_cast<int32_t>(i);
}

// The chunk's K/V rows to their slots: token i of sequence b sits at position
// L_b - n_b + i.  One thread per kAppendVec 16-byte chunks of a (token, kv
// head) row, so that each thread keeps several loads in flight behind its
// block-table read.  Block (0, num_seqs) orders the attention's work items
// instead.
__global__ void __launch_bounds__(kAppendThreads)
chunk_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ context_lens,
                    const int32_t* __restrict__ block_tables, int max_blocks, int block_size,
                    int64_t num_blocks, int num_kv_heads, int chunks_per_row,
                    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_seqs,
                    const PlanArgs pa) {
  pdl_launch_dependents();
  pdl_wait_prior();
  if (static_cast<int>(blockIdx.y) == num_seqs) {
    if (blockIdx.x == 0)
      plan_items(cu_q, context_lens, num_seqs, max_blocks, block_size, pa);
    return;
  }
  const int b = blockIdx.y;
  const int start = cu_q[b];
  const int n = cu_q[b + 1] - start;
  const int vecs_per_row = chunks_per_row / kAppendVec;
  const int64_t per_tok = static_cast<int64_t>(num_kv_heads) * vecs_per_row;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n * per_tok) return;
  const int i = static_cast<int>(idx / per_tok);
  const int rem = static_cast<int>(idx - i * per_tok);
  const int h = rem / vecs_per_row, c = (rem - h * vecs_per_row) * kAppendVec;
  // the rows' loads go out before the block-table read, not after it
  const int64_t src = (static_cast<int64_t>(start + i) * num_kv_heads + h) * chunks_per_row + c;
  uint4 kr[kAppendVec], vr[kAppendVec];
#pragma unroll
  for (int e = 0; e < kAppendVec; ++e) {
    kr[e] = __ldg(k + src + e);
    vr[e] = __ldg(v + src + e);
  }
  const int64_t p = static_cast<int64_t>(context_lens[b]) - n + i;
  if (p < 0 || p >= static_cast<int64_t>(max_blocks) * block_size) return;
  const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + p / block_size];
  if (blk < 0 || blk >= num_blocks) return;
  const int64_t dst = ((static_cast<int64_t>(blk) * num_kv_heads + h) * block_size +
                       p % block_size) * chunks_per_row + c;
#pragma unroll
  for (int e = 0; e < kAppendVec; ++e) {
    k_cache[dst + e] = kr[e];
    v_cache[dst + e] = vr[e];
  }
}

}  // namespace

cudaError_t launch_prefill(int dtype, int head_dim, const void* q, const void* k, const void* v,
                           const int32_t* cu_q, int num_seqs, int num_q_heads, int max_chunk,
                           void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads,
                           int block_size, const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, int window, int num_sinks, float scale,
                           void* out, int32_t* order, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream) {
  if (num_seqs == 0 || max_chunk == 0) return cudaSuccess;
  // 1) the chunk's rows to their slots; the work items' order
  const int cpr = head_dim * 2 / 16;
  const int64_t per_seq = static_cast<int64_t>(max_chunk) * num_kv_heads * (cpr / kAppendVec);
  PlanArgs pa;
  pa.order = order;
  pa.tok_per_cta = kPrefillRowsCta >> prefill_heads_log2(num_q_heads / num_kv_heads);
  pa.chunks_per_seq = (max_chunk + pa.tok_per_cta - 1) / pa.tok_per_cta;
  pa.window = window;
  pa.num_sinks = num_sinks;
  dim3 agrid(static_cast<unsigned>((per_seq + kAppendThreads - 1) / kAppendThreads),
             num_seqs + 1);
  cudaError_t e = launch_pdl(chunk_append_kernel, agrid, dim3(kAppendThreads), 0, stream,
                             static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_q,
                             context_lens, block_tables, max_blocks, block_size, num_blocks,
                             num_kv_heads, cpr, static_cast<uint4*>(k_cache),
                             static_cast<uint4*>(v_cache), num_seqs, pa);
  if (e != cudaSuccess) return e;
  // 2) attention over prefix + chunk on the tensor cores, items in that order
  return launch_prefill_tc(dtype, head_dim, q, cu_q, num_seqs, num_q_heads, max_chunk,
                           num_blocks, num_kv_heads, block_size, block_tables, max_blocks,
                           context_lens, window, num_sinks, scale, out, order, kmap, vmap,
                           stream);
}

}  // namespace pkv
