// pkv_prefill_tc.cu -- chunked prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// What is computed: see pkv_prefill.cu ("Building a Streaming Sliding-Window
// Attention Engine in Pure Python", Step 3, prefill_attention: query at
// position p attends keys j <= p with p - j < window, softmax per row).
//
// How: a CTA of 128 threads owns 128 query rows of one (sequence, kv head):
// (token, GQA head) pairs, so every K/V page read serves the whole group.
// Thread t owns row t, which is also TMEM lane t.  Per tile of 64 keys:
//   1. TMA brings the four 16-key K and V units of the tile (128-byte swizzle)
//      into one of two stages;
//   2. thread 0 issues S = Q K^T (M = 128, N = 64, K = head_dim; both operands
//      K-major in shared memory) into TMEM;
//   3. every thread loads its S row from TMEM and runs the online softmax on
//      it alone -- row maxima and sums need no shuffles;
//   4. P is written to shared memory as a K-major operand, split into a hi
//      and a lo 16-bit part (so the weights keep ~fp32 precision), and thread
//      0 issues O += P_hi V + P_lo V (N = head_dim, V read MN-major straight
//      from its TMA tile) into TMEM;
//   5. when a row's running maximum moves by more than 2^8, the row's O in
//      TMEM is rescaled in place (lazy rescaling).
// V rows of keys that no query of the CTA may see are zeroed before the
// products, so garbage (even NaN) in unused slots cannot leak.
#include <limits.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kTRows = 128;       // query rows per CTA == TMEM lanes
constexpr int kTKeys = 64;        // keys per tile
constexpr int kTUnits = kTKeys / kUnitTokens;
constexpr int kTThreads = 128;
constexpr float kTRescale = 8.0f;

struct TcParams {
  const void* q;
  void* out;
  const int32_t* cu_q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int64_t num_blocks;
  int num_q_heads, num_kv_heads, group;
  int head_chunk_log2, num_head_chunks;
  int max_blocks, block_size, window;
  int max_units;
  float scale_log2;
};

template <int D>
struct TcLayout {
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kKBlocks = D / 64;                  // 128-byte column blocks
  static constexpr int kQBytes = kKBlocks * kTRows * 128;
  static constexpr int kKVTile = kKBlocks * kTKeys * 128;  // K (or V) of one tile
  static constexpr int kStageBytes = 2 * kKVTile;
  static constexpr int kPBytes = kTRows * 128;             // 64 keys x 2 bytes per row
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQBytes;
  static constexpr int kPOff = kStageOff + kStages * kStageBytes;
  static constexpr int kYOff = kPOff + 2 * kPBytes;
  static constexpr uint32_t kTmemCols = (64 + D) <= 128 ? 128 : 256;  // S: 64, O: D
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <typename T, int D>
__global__ void __launch_bounds__(kTThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const TcParams p) {
  using Lay = TcLayout<D>;
  constexpr int S = Lay::kStages;
  constexpr uint32_t kFmt = __is_same(T, __nv_bfloat16) ? 1u : 0u;
  constexpr uint32_t kIdS = umma_idesc_f16(kFmt, kTRows, kTKeys, 0);
  constexpr uint32_t kIdO = umma_idesc_f16(kFmt, kTRows, D, 1);

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t s_bar, pv_bar, done_bar;
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait_prior();

  const int b = blockIdx.z;
  const int hkv = blockIdx.y / p.num_head_chunks;
  const int chunk = blockIdx.y - hkv * p.num_head_chunks;
  const int gc = 1 << p.head_chunk_log2;
  const int tok_per_cta = kTRows >> p.head_chunk_log2;
  const int start = p.cu_q[b];
  const int n = p.cu_q[b + 1] - start;
  const int tile0 = blockIdx.x * tok_per_cta;
  if (tile0 >= n) return;
  const int L = p.context_lens[b];
  const int tile_n = min(tok_per_cta, n - tile0);
  const int pos0 = L - n + tile0, pos1 = pos0 + tile_n - 1;
  const bool len_ok = L >= n && pos0 >= 0 &&
                      static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_blocks) * p.block_size;
  const int k_lo = (p.window > 0) ? max(0, pos0 - p.window + 1) : 0;
  const int u_first = k_lo / kUnitTokens;
  const int n_units = len_ok ? pos1 / kUnitTokens - u_first + 1 : 0;

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  int* ys = reinterpret_cast<int*>(smem_raw + (base - raw_addr) + Lay::kYOff);

  // ---- set-up: TMEM, barriers, page rows of the key range, the Q tile ----
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(Lay::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
    mbar_init(smem_u32(&s_bar), 1);
    mbar_init(smem_u32(&pv_bar), 1);
    mbar_init(smem_u32(&done_bar), 1);
    fence_mbar_init();
  }
  bool bad = !(len_ok && n_units <= p.max_units);
  const int n_load = min(n_units, p.max_units);
  for (int u = tid; u < n_load; u += kTThreads) {
    const int t0 = (u_first + u) * kUnitTokens;
    const int32_t pb = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks +
                             t0 / p.block_size);
    const bool ok = pb >= 0 && pb < p.num_blocks;
    ys[u] = ok ? (pb * p.num_kv_heads + hkv) * p.block_size + (t0 % p.block_size) : -1;
    if (!ok) bad = true;
  }
  // this thread's query row: token ti of the tile, head hi of the chunk
  const int ti = tid >> p.head_chunk_log2, hi = tid & (gc - 1);
  const bool row_ok = ti < tile_n;
  const int rpos = row_ok ? pos0 + ti : -1;
  {
    const uint4* qrow = reinterpret_cast<const uint4*>(
        static_cast<const T*>(p.q) +
        (static_cast<int64_t>(start + tile0 + (row_ok ? ti : 0)) * p.num_q_heads +
         hkv * p.group + chunk * gc + hi) * D);
#pragma unroll
    for (int c16 = 0; c16 < D / 8; ++c16) {
      const uint4 v = row_ok ? __ldg(qrow + c16) : make_uint4(0u, 0u, 0u, 0u);
      st_shared_v4(base + Lay::kQOff + (c16 >> 3) * kTRows * 128 + sw128(tid, c16), v);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  const bool bad_cta = __syncthreads_or(bad) != 0;
  tc_fence_after();
  bad = bad_cta;
  const uint32_t tmem = tmem_base_s;
  const uint32_t tS = tmem, tO = tmem + 64;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const int n_tiles = bad_cta ? 0 : (n_units + kTUnits - 1) / kTUnits;

  // TMA of the units of tile j that exist (thread 0 only)
  auto issue = [&](int j) {
    const int stage = j % S;
    const uint32_t bar = smem_u32(&full_bar[stage]);
    const uint32_t kdst = base + Lay::kStageOff + stage * Lay::kStageBytes;
    const uint32_t vdst = kdst + Lay::kKVTile;
    const int units = min(kTUnits, n_units - j * kTUnits);
    mbar_arrive_expect_tx(bar, units * 2 * Lay::kKBlocks * kUnitTokens * 128);
    for (int i = 0; i < units; ++i) {
      const int y = ys[j * kTUnits + i];
#pragma unroll
      for (int kb = 0; kb < Lay::kKBlocks; ++kb) {
        const uint32_t off = kb * kTKeys * 128 + i * kUnitTokens * 128;
        tma_load_2d(kdst + off, &kmap, kb * 64, y, bar);
        tma_load_2d(vdst + off, &vmap, kb * 64, y, bar);
      }
    }
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < min(S, n_tiles); ++issued) issue(issued);

  float m_run = -INFINITY, l_run = 0.f;
  const uint32_t ph = base + Lay::kPOff, pl = ph + Lay::kPBytes;
  int j = 0;
  for (; j < n_tiles; ++j) {
    const int stage = j % S;
    const uint32_t kst = base + Lay::kStageOff + stage * Lay::kStageBytes;
    const uint32_t vst = kst + Lay::kKVTile;
    const int t0 = (u_first + j * kTUnits) * kUnitTokens;
    if (!mbar_wait_bounded(smem_u32(&full_bar[stage]), (j / S) & 1, kWaitLimit)) bad = true;

    // ---- S = Q K^T into TMEM columns [0, 64) ----
    // (every thread read S(j-1) before the last barrier, so it may be overwritten)
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t ad =
            umma_sdesc_sw128(base + Lay::kQOff + (kk >> 2) * kTRows * 128 + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = umma_sdesc_sw128(kst + (kk >> 2) * kTKeys * 128 + (kk & 3) * 32, 16, 1024);
        umma_f16(tS, ad, bd, kIdS, kk > 0 ? 1u : 0u);
      }
      umma_commit(smem_u32(&s_bar));
    }

    // V rows of keys outside [k_lo, pos1] (before the window of every row, past
    // the chunk, or never loaded) may hold anything, even NaN: zero them so that
    // their zero weights give exact zeros
    if ((t0 < k_lo || t0 + kTKeys - 1 > pos1) && tid < kTKeys) {
      const int kp = t0 + tid;
      if (kp < k_lo || kp > pos1) {
#pragma unroll
        for (int kb = 0; kb < Lay::kKBlocks; ++kb)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(vst + kb * kTKeys * 128 + tid * 128 + c * 16, make_uint4(0u, 0u, 0u, 0u));
      }
    }

    if (!mbar_wait_bounded(smem_u32(&s_bar), j & 1, kWaitLimit)) bad = true;
    tc_fence_after();

    // ---- the row's scores: mask, log2 scale, maximum ----
    float s[kTKeys];
#pragma unroll
    for (int c = 0; c < kTKeys; c += 16) {
      float v[16];
      tmem_ld16(tS + lane_off + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) s[c + i] = v[i];
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kTKeys; ++c) {
      const int kp = t0 + c;
      const bool valid = kp <= rpos && (p.window <= 0 || rpos - kp < p.window);
      s[c] = valid ? s[c] * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, s[c]);
    }
    const float m_old = m_run;
    const bool need = mx > m_old + kTRescale;
    if (need) m_run = mx;
    const bool rescale = need && m_old != -INFINITY;
    const float alpha = rescale ? ex2(m_old - m_run) : 1.f;
    l_run *= alpha;

    // P and O are free once the previous PV product completed; so is the stage
    // tile j-1 used, which takes tile j-1+S
    if (j > 0) {
      if (!mbar_wait_bounded(smem_u32(&pv_bar), (j - 1) & 1, kWaitLimit)) bad = true;
      tc_fence_after();
      if (tid == 0 && issued < n_tiles && !bad) issue(issued++);
    }

    // ---- P rows (hi, lo) as K-major operands ----
#pragma unroll
    for (int c8 = 0; c8 < kTKeys / 8; ++c8) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = ex2(s[c8 * 8 + 2 * e] - m_run);
        const float p1 = ex2(s[c8 * 8 + 2 * e + 1] - m_run);
        l_run += p0 + p1;
        hw[e] = Mma<T>::pack(p0, p1);
        lw[e] = Mma<T>::pack(p0 - Mma<T>::lo_f32(hw[e]), p1 - Mma<T>::hi_f32(hw[e]));
      }
      st_shared_v4(ph + sw128(tid, c8), make_uint4(hw[0], hw[1], hw[2], hw[3]));
      st_shared_v4(pl + sw128(tid, c8), make_uint4(lw[0], lw[1], lw[2], lw[3]));
    }
    // ---- lazy rescale of the row's O (after PV(j-1), before PV(j)) ----
    if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float v[16];
        tmem_ld16(tO + lane_off + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= alpha;
        tmem_st16(tO + lane_off + c, v);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
    tc_fence_after();

    // ---- O += P_hi V + P_lo V into TMEM columns [64, 64 + D) ----
    if (tid == 0) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int kk = 0; kk < kTKeys / 16; ++kk) {
          const uint64_t ad = umma_sdesc_sw128((part ? pl : ph) + kk * 32, 16, 1024);
          // V: keys are the K dimension (8-row groups 1 KB apart, 16 keys per
          // step), head dims the N dimension (64-column blocks one tile apart)
          const uint64_t bd = umma_sdesc_sw128(vst + kk * 16 * 128, kTKeys * 128, 1024);
          umma_f16(tO, ad, bd, kIdO, (j > 0 || kk > 0 || part > 0) ? 1u : 0u);
        }
      }
      umma_commit(smem_u32(&pv_bar));
    }
  }

  // ---- drain: every product and every copy this CTA started has landed ----
  // (products were issued iff there was a tile)
  if (tid == 0) {
    if (n_tiles > 0) umma_commit(smem_u32(&done_bar));
    for (int t = j; t < issued; ++t)
      if (!mbar_wait_bounded(smem_u32(&full_bar[t % S]), (t / S) & 1, kWaitLimit)) bad = true;
  }
  if (n_tiles > 0 && !mbar_wait_bounded(smem_u32(&done_bar), 0, kWaitLimit)) bad = true;
  tc_fence_after();
  const bool nan_out = __syncthreads_or(bad) != 0;

  // ---- epilogue: O / l to the output rows (TMEM loads are warp-wide) ----
  T* dst = static_cast<T*>(p.out) +
           (static_cast<int64_t>(start + tile0 + (row_ok ? ti : 0)) * p.num_q_heads +
            hkv * p.group + chunk * gc + hi) * D;
  const float inv = nan_out ? __int_as_float(0x7fc00000) : 1.f / l_run;
#pragma unroll
  for (int c = 0; c < D; c += 16) {
    float v[16];
    if (!nan_out) {
      tmem_ld16(tO + lane_off + c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    }
    if (row_ok) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = Mma<T>::pack(v[2 * i] * inv, v[2 * i + 1] * inv);
      reinterpret_cast<uint4*>(dst + c)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dst + c)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(Lay::kTmemCols));
}

template <typename T, int D>
cudaError_t launch_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const TcParams& p,
                     int max_chunk, int num_seqs, cudaStream_t stream) {
  using Lay = TcLayout<D>;
  auto kern = prefill_tc_kernel<T, D>;
  const size_t smem = 1024 + Lay::kYOff + sizeof(int) * p.max_units;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tok_per_cta = kTRows >> p.head_chunk_log2;
  dim3 grid((max_chunk + tok_per_cta - 1) / tok_per_cta, p.num_kv_heads * p.num_head_chunks,
            num_seqs);
  return launch_pdl(kern, grid, dim3(kTThreads), smem, stream, kmap, vmap, p);
}

}  // namespace

size_t prefill_tc_smem_bytes(int head_dim, int max_units) {
  const int y = head_dim == 128 ? TcLayout<128>::kYOff : TcLayout<64>::kYOff;
  return 1024 + y + sizeof(int) * static_cast<size_t>(max_units);
}

cudaError_t launch_prefill_tc(int dtype, int head_dim, const void* q, const int32_t* cu_q,
                              int num_seqs, int num_q_heads, int max_chunk, int64_t num_blocks,
                              int num_kv_heads, int block_size, const int32_t* block_tables,
                              int max_blocks, const int32_t* context_lens, int window,
                              float scale, void* out, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t stream) {
  TcParams p{};
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
  while (gc * 2 <= 16 && p.group % (gc * 2) == 0) gc *= 2;
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
    if (head_dim == 128) return launch_t<__half, 128>(kmap, vmap, p, max_chunk, num_seqs, stream);
    return launch_t<__half, 64>(kmap, vmap, p, max_chunk, num_seqs, stream);
  }
  if (head_dim == 128)
    return launch_t<__nv_bfloat16, 128>(kmap, vmap, p, max_chunk, num_seqs, stream);
  return launch_t<__nv_bfloat16, 64>(kmap, vmap, p, max_chunk, num_seqs, stream);
}

}  // namespace pkv
