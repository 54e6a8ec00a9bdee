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

// bf16 caches: blocks that record the range of V magnitudes of each
// (sequence, kv head) over its context, one partial per block of scan_rows
// context rows: vparts[pair * row_blocks + rb] = (largest magnitude, smallest
// non-zero magnitude minus one), as bf16 bits ((0, 0xffffffff) for no rows).
struct ScanArgs {
  uint2* vparts;  // nullptr: no scan (fp16 caches)
  const uint4* v_cache;
  int row_blocks, scan_rows;
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

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t add_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One scan block: rows rb * scan_rows .. of sequence b, kv head h.  Rows of
// the cached prefix come from the pool, the chunk's rows from the input v
// (the append blocks write them to the pool at the same time).  Each thread
// takes one 16-byte column chunk of several rows, reading the rows' block-table
// entries first and then all their values, so both reads overlap.
__device__ void scan_v_range(const uint4* __restrict__ v, const int32_t* __restrict__ cu_q,
                             const int32_t* __restrict__ context_lens,
                             const int32_t* __restrict__ block_tables, int max_blocks,
                             int block_size, int64_t num_blocks, int num_kv_heads,
                             int chunks_per_row, int b, int h, int rb, const ScanArgs& sa) {
  constexpr int kRowsPerThread = 8;
  __shared__ uint32_t red[2][kAppendThreads / 32];
  const int tid = threadIdx.x;
  const int start = cu_q[b], n = cu_q[b + 1] - start;
  const int L = context_lens[b];
  const bool ok = L >= n && static_cast<int64_t>(L) <= static_cast<int64_t>(max_blocks) * block_size;
  const int r_begin = rb * sa.scan_rows, r_end = ok ? min(L, r_begin + sa.scan_rows) : 0;
  const int rows_per_pass = kAppendThreads / chunks_per_row;
  const int c = tid % chunks_per_row;
  uint32_t mx = 0u, mn = 0xffffffffu;  // per bf16 half: max magnitude, min (magnitude - 1)
  for (int r0 = r_begin + tid / chunks_per_row; r0 < r_end; r0 += kRowsPerThread * rows_per_pass) {
    int64_t src[kRowsPerThread];
#pragma unroll
    for (int e = 0; e < kRowsPerThread; ++e) {
      const int r = r0 + e * rows_per_pass;
      src[e] = -1;
      if (r >= r_end) continue;
      if (r >= L - n) {
        src[e] = -2 - ((static_cast<int64_t>(start) + r - (L - n)) * num_kv_heads + h);
      } else {
        const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + r / block_size];
        if (blk >= 0 && blk < num_blocks)
          src[e] = (static_cast<int64_t>(blk) * num_kv_heads + h) * block_size + r % block_size;
      }
    }
    uint4 x[kRowsPerThread];
#pragma unroll
    for (int e = 0; e < kRowsPerThread; ++e) {
      x[e] = make_uint4(0u, 0u, 0u, 0u);
      if (src[e] >= 0)
        x[e] = sa.v_cache[src[e] * chunks_per_row + c];
      else if (src[e] <= -2)
        x[e] = __ldg(v + (-2 - src[e]) * chunks_per_row + c);
    }
#pragma unroll
    for (int e = 0; e < kRowsPerThread; ++e) {
      if (src[e] == -1) continue;
      const uint32_t w[4] = {x[e].x, x[e].y, x[e].z, x[e].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t a = w[q] & 0x7fff7fffu;
        mx = max_u16x2(mx, a);
        mn = min_u16x2(mn, add_u16x2(a, 0xffffffffu));  // a zero wraps to 0xffff
      }
    }
  }
  uint32_t m1 = max(mx & 0xffffu, mx >> 16), m2 = min(mn & 0xffffu, mn >> 16);
  m1 = __reduce_max_sync(0xffffffffu, m1);
  m2 = __reduce_min_sync(0xffffffffu, m2);
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = m1;
    red[1][tid >> 5] = m2;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kAppendThreads / 32; ++w) {
      m1 = max(m1, red[0][w]);
      m2 = min(m2, red[1][w]);
    }
    if (m1 == 0u) m2 = 0xffffffffu;  // nothing non-zero
    sa.vparts[(static_cast<int64_t>(b) * num_kv_heads + h) * sa.row_blocks + rb] = make_uint2(m1, m2);
  }
}

// The chunk's K/V rows to their slots: token i of sequence b sits at position
// L_b - n_b + i.  One thread per kAppendVec 16-byte chunks of a (token, kv
// head) row, so that each thread keeps several loads in flight behind its
// block-table read.  Block (0, num_seqs) orders the attention's work items
// instead; blocks (append_blocks + h * row_blocks + rb, b) scan V ranges.
__global__ void __launch_bounds__(kAppendThreads)
chunk_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ context_lens,
                    const int32_t* __restrict__ block_tables, int max_blocks, int block_size,
                    int64_t num_blocks, int num_kv_heads, int chunks_per_row,
                    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_seqs,
                    int append_blocks, const PlanArgs pa, const ScanArgs sa) {
  pdl_launch_dependents();
  pdl_wait_prior();
  if (static_cast<int>(blockIdx.y) == num_seqs) {
    if (blockIdx.x == 0)
      plan_items(cu_q, context_lens, num_seqs, max_blocks, block_size, pa);
    return;
  }
  const int b = blockIdx.y;
  if (static_cast<int>(blockIdx.x) >= append_blocks) {
    const int s = static_cast<int>(blockIdx.x) - append_blocks;
    scan_v_range(v, cu_q, context_lens, block_tables, max_blocks, block_size, num_blocks,
                 num_kv_heads, chunks_per_row, b, s / sa.row_blocks, s % sa.row_blocks, sa);
    return;
  }
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
                           void* out, int32_t* order, uint2* vparts, uint32_t* mode,
                           const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream) {
  if (num_seqs == 0 || max_chunk == 0) return cudaSuccess;
  // 1) the chunk's rows to their slots; the work items' order; (bf16) the V ranges
  const int cpr = head_dim * 2 / 16;
  const int64_t per_seq = static_cast<int64_t>(max_chunk) * num_kv_heads * (cpr / kAppendVec);
  PlanArgs pa;
  pa.order = order;
  pa.tok_per_cta = kPrefillRowsCta >> prefill_heads_log2(num_q_heads / num_kv_heads);
  pa.chunks_per_seq = (max_chunk + pa.tok_per_cta - 1) / pa.tok_per_cta;
  pa.window = window;
  pa.num_sinks = num_sinks;
  ScanArgs sa{};
  const PrefillScan plan = prefill_scan_plan(max_blocks, block_size);
  if (dtype == 2) {
    sa.vparts = vparts;
    sa.v_cache = static_cast<const uint4*>(v_cache);
    sa.row_blocks = plan.row_blocks;
    sa.scan_rows = plan.scan_rows;
  }
  const int64_t append_blocks = (per_seq + kAppendThreads - 1) / kAppendThreads;
  const int64_t gx = append_blocks + (sa.vparts ? static_cast<int64_t>(num_kv_heads) * sa.row_blocks : 0);
  if (gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 agrid(static_cast<unsigned>(gx), num_seqs + 1);
  cudaError_t e = launch_pdl(chunk_append_kernel, agrid, dim3(kAppendThreads), 0, stream,
                             static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_q,
                             context_lens, block_tables, max_blocks, block_size, num_blocks,
                             num_kv_heads, cpr, static_cast<uint4*>(k_cache),
                             static_cast<uint4*>(v_cache), num_seqs,
                             static_cast<int>(append_blocks), pa, sa);
  if (e != cudaSuccess) return e;
  // 2) attention over prefix + chunk on the tensor cores, items in that order
  return launch_prefill_tc(dtype, head_dim, q, cu_q, num_seqs, num_q_heads, max_chunk,
                           num_blocks, num_kv_heads, block_size, block_tables, max_blocks,
                           context_lens, window, num_sinks, scale, out, order, vparts,
                           plan.row_blocks, mode, kmap, vmap, stream);
}

}  // namespace pkv
