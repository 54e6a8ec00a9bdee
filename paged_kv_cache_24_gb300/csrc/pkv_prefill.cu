// pkv_prefill.cu -- paged chunked prefill.
//
// What is computed ("Building a Streaming Sliding-Window Attention Engine in
// Pure Python", Step 3, prefill_attention: the mask (i - j) < window and
// j <= i, softmax per query row): sequence b holds L_b tokens after a chunk of
// n_b new ones was appended at positions L_b - n_b .. L_b - 1; the query of
// the chunk token at position p attends positions j <= p (and p - j < window
// when window > 0) of the paged cache -- the cached prefix and the chunk.
//
// How: the chunk's K/V rows are first written to their slots (one kernel),
// then an attention kernel treats (query token, query head) pairs as the rows
// of a dense tile: 64 rows per CTA (4 warps x 16), the GQA heads of a token
// side by side so they share every K/V page.  Pages stream through a
// CTA-shared ring of TMA stages (full barrier: transaction bytes; empty
// barrier: one arrival per warp).  S = Q K^T and O += P V run on the tensor
// cores (mma.m16n8k16, fp32 accumulate); the accumulator of S is already the
// A fragment of P, so no data moves between the two products.  P is carried as
// a hi + lo pair of 16-bit values, the softmax is online in fp32.
#include <limits.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPWarps = 4;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPRows = 16 * kPWarps;  // query rows per CTA
constexpr int kPStages = 4;
constexpr int kBox = kUnitTokens * 128;  // one TMA box: 16 rows x 128 bytes
constexpr float kPRescale = 8.0f;

__device__ __forceinline__ uint32_t pswz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * kBox + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

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

struct PrefillParams {
  const void* q;              // [T][Hq][D]
  void* out;                  // [T][Hq][D]
  const int32_t* cu_q;        // [B+1]
  const int32_t* block_tables;
  const int32_t* context_lens;
  int64_t num_blocks;
  int num_q_heads, num_kv_heads, group;
  int head_chunk_log2;        // query heads per CTA = 1 << head_chunk_log2 (<= 16)
  int num_head_chunks;
  int max_blocks, block_size, window;
  int max_units;              // capacity of the shared page-row table
  float scale_log2;
};

template <typename T, int D>
__global__ void __launch_bounds__(kPThreads, 2)
prefill16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const PrefillParams p) {
  constexpr int KS = D / 16;          // k-steps of Q K^T
  constexpr int NTD = D / 8;          // n-tiles of O (8 head dims each)
  constexpr int kBoxes = D / 64;
  constexpr int kTile = kBoxes * kBox;
  constexpr int kStage = 2 * kTile;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kPStages];
  __shared__ __align__(8) uint64_t empty_bar[kPStages];
  __shared__ int s_bad;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  pdl_launch_dependents();
  pdl_wait_prior();

  const int b = blockIdx.z;
  const int hkv = blockIdx.y / p.num_head_chunks;
  const int chunk = blockIdx.y - hkv * p.num_head_chunks;
  const int gc = 1 << p.head_chunk_log2;          // heads per token row group
  const int tok_per_cta = kPRows >> p.head_chunk_log2;
  const int start = p.cu_q[b];
  const int n = p.cu_q[b + 1] - start;
  const int tile0 = blockIdx.x * tok_per_cta;     // first chunk token of this CTA
  if (tile0 >= n) return;
  const int L = p.context_lens[b];
  const int tile_n = min(tok_per_cta, n - tile0);
  const int pos0 = L - n + tile0;                 // position of the CTA's first token
  const int pos1 = pos0 + tile_n - 1;             // and of its last
  const bool len_ok = L >= n && pos0 >= 0 &&
                      static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_blocks) * p.block_size;
  const int k_lo = (p.window > 0) ? max(0, pos0 - p.window + 1) : 0;
  const int u_first = k_lo / kUnitTokens;
  const int n_units = len_ok ? pos1 / kUnitTokens - u_first + 1 : 0;

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  int* ys = reinterpret_cast<int*>(smem_raw + (base_addr - raw_addr) + kPStages * kStage);

  // ---- set-up: barriers, page rows of every unit of the key range ----
  if (threadIdx.x == 0) {
    s_bad = (len_ok && n_units <= p.max_units) ? 0 : 1;
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kPWarps);
    }
    fence_mbar_init();
  }
  const int n_load = min(n_units, p.max_units);
  for (int u = threadIdx.x; u < n_load; u += kPThreads) {
    const int t0 = (u_first + u) * kUnitTokens;
    const int32_t pb = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks +
                             t0 / p.block_size);
    ys[u] = (pb >= 0 && pb < p.num_blocks)
                ? (pb * p.num_kv_heads + hkv) * p.block_size + (t0 % p.block_size)
                : -1;
  }
  __syncthreads();
  const bool bad_cta = s_bad != 0;
  const int units = bad_cta ? 0 : n_units;

  auto issue = [&](int j) {
    const int stage = j % kPStages;
    const uint32_t bar = smem_u32(&full_bar[stage]);
    const uint32_t kdst = base_addr + stage * kStage;
    const int y = ys[j];
    if (y >= 0) {
      mbar_arrive_expect_tx(bar, kStage);
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_load_2d(kdst + bx * kBox, &kmap, bx * 64, y, bar);
        tma_load_2d(kdst + kTile + bx * kBox, &vmap, bx * 64, y, bar);
      }
    } else {
      mbar_arrive(bar);
    }
  };
  if (threadIdx.x == 0)
    for (int j = 0; j < min(kPStages, units); ++j) issue(j);

  // ---- this warp's 16 query rows: row r = (token r / gc, head r % gc) ----
  int rpos[2];          // positions of rows g and g + 8 (-1: no such row)
  uint32_t qa[KS][4];   // Q A fragments
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = warp * 16 + g + 8 * half;
    const int ti = r >> p.head_chunk_log2, hi = r & (gc - 1);
    const bool ok = ti < tile_n && chunk * gc + hi < p.group;
    rpos[half] = ok ? pos0 + ti : -1;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(p.q) +
        (static_cast<int64_t>(start + tile0 + ti) * p.num_q_heads + hkv * p.group + chunk * gc +
         hi) * D);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qa[kk][half] = ok ? __ldg(qrow + kk * 8 + tig) : 0u;          // d = 16kk + 2tig
      qa[kk][2 + half] = ok ? __ldg(qrow + kk * 8 + 4 + tig) : 0u;  // d + 8
    }
  }
  const int wpos_min = min(rpos[0] < 0 ? INT_MAX : rpos[0], rpos[1] < 0 ? INT_MAX : rpos[1]);

  float o[NTD][4];
#pragma unroll
  for (int i = 0; i < NTD; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) o[i][r] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  bool bad = bad_cta;

  for (int j = 0; j < units; ++j) {
    const int stage = j % kPStages;
    const uint32_t parity = (j / kPStages) & 1;
    const bool ok = mbar_wait_bounded(smem_u32(&full_bar[stage]), parity, kWaitLimit);
    if (!__all_sync(0xffffffffu, ok)) {
      bad = true;
      break;
    }
    if (ys[j] < 0) bad = true;
    const uint32_t kt = base_addr + stage * kStage;
    const uint32_t vt = kt + kTile;
    const int t0 = (u_first + j) * kUnitTokens;

    // ---- S[16 rows x 16 keys] = Q K^T ----
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) s[nt][r] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t b0, b1, b2, b3;  // (keys 0-7 | 8-15) x (d 16kk.. | 16kk+8..)
      const int key = (lane & 7) + ((lane >> 4) << 3);
      ldmatrix_x4(kt + pswz(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
      Mma<T>::run(s[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
      Mma<T>::run(s[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
    }

    // ---- mask (causal, window), log2 scale, row maxima ----
    const bool full = t0 + kUnitTokens - 1 <= wpos_min && rpos[0] >= 0 && rpos[1] >= 0 &&
                      (p.window <= 0 || max(rpos[0], rpos[1]) - t0 < p.window);
    float mx[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = s[nt][2 * half + e] * p.scale_log2;
          if (!full) {
            const int kp = t0 + nt * 8 + 2 * tig + e;
            const int rp = rpos[half];
            const bool valid = rp >= 0 && kp <= rp && (p.window <= 0 || rp - kp < p.window);
            x = valid ? x : -INFINITY;
          }
          s[nt][2 * half + e] = x;
          v = fmaxf(v, x);
        }
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      mx[half] = v;
    }
    const bool need = (mx[0] > m_run[0] + kPRescale) || (mx[1] > m_run[1] + kPRescale);
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float mnew = mx[half] > m_run[half] + kPRescale ? mx[half] : m_run[half];
        const float alpha = (m_run[half] == -INFINITY) ? 0.f : ex2(m_run[half] - mnew);
        m_run[half] = mnew;
        l_run[half] *= alpha;
#pragma unroll
        for (int i = 0; i < NTD; ++i) {
          o[i][2 * half] *= alpha;
          o[i][2 * half + 1] *= alpha;
        }
      }
    }
    // ---- P = 2^(s - m): hi + lo 16-bit A fragments (rows g, g+8; keys 0-7, 8-15) ----
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float m = m_run[half];
        const float p0 = (m == -INFINITY) ? 0.f : ex2(s[nt][2 * half] - m);
        const float p1 = (m == -INFINITY) ? 0.f : ex2(s[nt][2 * half + 1] - m);
        l_run[half] += p0 + p1;
        const uint32_t h = Mma<T>::pack(p0, p1);
        ph[2 * nt + half] = h;
        pl[2 * nt + half] = Mma<T>::pack(p0 - Mma<T>::lo_f32(h), p1 - Mma<T>::hi_f32(h));
      }
    // keys outside [k_lo, pos1] may hold anything (even NaN): zero their V rows
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (t0 < k_lo || t0 + kUnitTokens - 1 > pos1) {
      const int kp = t0 + 2 * tig;
      mlo = ((kp >= k_lo && kp <= pos1) ? 0x0000ffffu : 0u) |
            ((kp + 1 >= k_lo && kp + 1 <= pos1) ? 0xffff0000u : 0u);
      mhi = ((kp + 8 >= k_lo && kp + 8 <= pos1) ? 0x0000ffffu : 0u) |
            ((kp + 9 >= k_lo && kp + 9 <= pos1) ? 0xffff0000u : 0u);
    }
    // ---- O[16 x D] += P[16 x 16] V[16 x D] ----
#pragma unroll
    for (int c = 0; c < NTD; c += 2) {
      uint32_t v0, v1, v2, v3;  // (keys 0-7 | 8-15) x (d tile c | c+1)
      const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
      ldmatrix_x4_trans(vt + pswz(key, c + (lane >> 4)), v0, v1, v2, v3);
      v0 &= mlo;
      v1 &= mhi;
      v2 &= mlo;
      v3 &= mhi;
      Mma<T>::run(o[c], ph[0], ph[1], ph[2], ph[3], v0, v1);
      Mma<T>::run(o[c], pl[0], pl[1], pl[2], pl[3], v0, v1);
      Mma<T>::run(o[c + 1], ph[0], ph[1], ph[2], ph[3], v2, v3);
      Mma<T>::run(o[c + 1], pl[0], pl[1], pl[2], pl[3], v2, v3);
    }

    // ---- release the stage; warp 0 refills it once every warp has ----
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
    if (warp == 0 && j + kPStages < units) {
      const bool freed =
          mbar_wait_bounded(smem_u32(&empty_bar[stage]), (j / kPStages) & 1, kWaitLimit);
      if (!__all_sync(0xffffffffu, freed)) {
        bad = true;
        break;
      }
      if (lane == 0) issue(j + kPStages);
    }
  }

  // ---- epilogue: normalise and store the valid rows ----
  if (bad) s_bad = 1;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float v = l_run[half];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    l_run[half] = v;
  }
  __syncthreads();
  const bool nan_out = s_bad != 0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (rpos[half] < 0) continue;
    const int r = warp * 16 + g + 8 * half;
    const int ti = r >> p.head_chunk_log2, hi = r & (gc - 1);
    T* dst = static_cast<T*>(p.out) +
             (static_cast<int64_t>(start + tile0 + ti) * p.num_q_heads + hkv * p.group +
              chunk * gc + hi) * D;
    const float inv = nan_out ? __int_as_float(0x7fc00000) : 1.f / l_run[half];
#pragma unroll
    for (int i = 0; i < NTD; ++i) {
      const uint32_t pk = Mma<T>::pack(o[i][2 * half] * inv, o[i][2 * half + 1] * inv);
      *reinterpret_cast<uint32_t*>(dst + i * 8 + 2 * tig) = pk;
    }
  }
}

template <typename T, int D>
cudaError_t launch_prefill_t(const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const PrefillParams& p, int max_chunk, int num_seqs,
                             cudaStream_t stream) {
  auto kern = prefill16_kernel<T, D>;
  const size_t smem = 1024 + kPStages * 2 * (D / 64) * kBox + sizeof(int) * p.max_units;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tok_per_cta = kPRows >> p.head_chunk_log2;
  dim3 grid((max_chunk + tok_per_cta - 1) / tok_per_cta, p.num_kv_heads * p.num_head_chunks,
            num_seqs);
  return launch_pdl(kern, grid, dim3(kPThreads), smem, stream, kmap, vmap, p);
}

}  // namespace

cudaError_t launch_prefill(int dtype, int head_dim, const void* q, const void* k, const void* v,
                           const int32_t* cu_q, int num_seqs, int num_q_heads, int max_chunk,
                           void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads,
                           int block_size, const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, int window, float scale, void* out,
                           const CUtensorMap& kmap, const CUtensorMap& vmap, bool tensor_memory,
                           cudaStream_t stream) {
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
  // 2) attention over prefix + chunk
  if (tensor_memory)
    return launch_prefill_tc(dtype, head_dim, q, cu_q, num_seqs, num_q_heads, max_chunk,
                             num_blocks, num_kv_heads, block_size, block_tables, max_blocks,
                             context_lens, window, scale, out, kmap, vmap, stream);
  PrefillParams p{};
  p.q = q;
  p.out = out;
  p.cu_q = cu_q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.num_blocks = num_blocks;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  int gc = 1;
  while (gc * 2 <= 16 && p.group % (gc * 2) == 0) gc *= 2;  // largest power of two dividing G
  int lg = 0;
  while ((1 << lg) < gc) ++lg;
  p.head_chunk_log2 = lg;
  p.num_head_chunks = p.group / gc;
  p.max_blocks = max_blocks;
  p.block_size = block_size;
  p.window = window;
  p.max_units = static_cast<int>(static_cast<int64_t>(max_blocks) * block_size / kUnitTokens) + 1;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (dtype == 1) {
    if (head_dim == 128) return launch_prefill_t<__half, 128>(kmap, vmap, p, max_chunk, num_seqs, stream);
    return launch_prefill_t<__half, 64>(kmap, vmap, p, max_chunk, num_seqs, stream);
  }
  if (head_dim == 128)
    return launch_prefill_t<__nv_bfloat16, 128>(kmap, vmap, p, max_chunk, num_seqs, stream);
  return launch_prefill_t<__nv_bfloat16, 64>(kmap, vmap, p, max_chunk, num_seqs, stream);
}

}  // namespace pkv
