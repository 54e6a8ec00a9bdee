// pkv_decode.cu -- single-query decode attention over a paged K/V pool.
//
// What is computed ("Build a Paged KV Cache in Pure Python", Step 4,
// scaled_dot_product_attention; "Building a Streaming Sliding-Window
// Attention Engine in Pure Python", Step 3, sliding_window_attention): for
// each sequence b and query head h (kv head h / G),
//     out = sum_t softmax_t(scale * q . K_t) V_t,   t in [lo, L),
// with K_t, V_t found through the block table (Step 3, retrieve).
//
// How (GB300 design):
//  * Work item = (sequence, kv head, head chunk, context split).  One CTA of
//    four warps per item; the split covers a fixed number of 16-token units
//    so every CTA streams the same number of bytes (flash-decoding split-K).
//  * Each warp owns a ring of shared-memory stages.  The warp resolves its
//    units' pages through the block table 32 at a time (one lane per unit),
//    and lane 0 issues one TMA tile load (cp.async.bulk.tensor, 128-byte
//    swizzle) for the unit's K rows and one for its V rows straight from the
//    page; completion arrives on the stage's mbarrier.  Nothing is gathered
//    through registers.
//  * 16-bit pools: S^T = K Q^T and O^T += V^T P^T on the tensor cores
//    (mma.m16n8k16, fp32 accumulate): 16 context tokens form the M side, the
//    G query heads of the group (padded to 8) the N side, so one page read
//    serves the whole GQA group.  P is carried as a hi + lo pair of 16-bit
//    values, so the weights keep ~fp32 precision.  The softmax is online in
//    fp32 (log2 domain), with lazy rescaling of the accumulator.
//  * fp32 pools: the same split structure on CUDA cores (float4 loads,
//    shuffle reductions).
//  * Every CTA ends with a cross-warp merge; a sequence with one split writes
//    its output directly, otherwise the unnormalised partial (m, l, o) goes to
//    the workspace and the combine kernel applies the log-sum-exp merge.
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// 4-byte asynchronous copy global -> shared through the load/store path,
// tracked by commit groups.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// wait until at most N of this thread's commit groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 3-D tiled load of the box at (x, y, z) into shared memory; completion is
// signalled as transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

constexpr int kThreads = kDecodeWarps * 32;
constexpr int kBoxBytes = kUnitTokens * 128;  // one TMA box: 16 rows x 128 bytes
constexpr float kRescaleThreshold = 8.0f;     // log2 units: weights stay <= 2^8

// Shared-memory plan of the tensor-core decode kernel.
//  16-bit pools: each warp's ring stage holds a unit's K and V tiles (16 rows
//    x D, 128-byte swizzled boxes), read by ldmatrix in place.
//  FP8 pools (KV8): a stage holds the unit's K and V code tiles (16 rows x D
//    bytes, one swizzled box each); the 2 x 16 row scales sit in a separate
//    per-warp array, filled by per-lane cp.async.  ldmatrix reads the codes
//    in place and the warp turns them into fp16 fragments in registers.
// kShallow: two ring stages per warp (16-bit pools, D = 128), so that three
// CTAs fit on an SM instead of two.  W: warps per CTA (each with its ring).
template <int D, bool KV8, bool kShallow = false, int W = kDecodeWarps>
struct Tile16 {
  static constexpr int kBoxes = D / 64;                     // 64 16-bit columns per box
  static constexpr int kTileBytes = kBoxes * kBoxBytes;     // fp16 K (or V) rows of one unit
  static constexpr int kCodeTileBytes = KV8 ? D * kUnitTokens : 0;
  static constexpr int kStageBytes = KV8 ? 2 * kCodeTileBytes : 2 * kTileBytes;
  static constexpr int kStages =
      KV8 ? kStagesFp8 : (kShallow ? 2 : (D == 128 ? kStagesD128 : kStagesD64));
  static constexpr int kRingBytes = kStages * kStageBytes;  // per warp
  static constexpr int kWarpBytes = kRingBytes;             // multiple of 1 KB
  static constexpr int kScaleBytes = KV8 ? kStages * 2 * kUnitTokens * 4 : 0;  // per warp
  static constexpr int kTxBytes = KV8 ? 2 * kCodeTileBytes : kStageBytes;  // TMA bytes per stage
  static constexpr int kSmemBytes = W * (kWarpBytes + kScaleBytes) + 1024;
  static_assert(kWarpBytes % 1024 == 0, "swizzled tiles need 1 KB alignment");
};

// Head-dim index of accumulator element r of m-tile mt held by lane group g.
//  16-bit pools: m-tile mt covers d = 16 mt .. 16 mt + 15 in order.
//  FP8 pools: m-tiles come in even / odd pairs over 32 d values: tile 2c + e
//  holds d = 32 c + e + 2 g (rows g) and 32 c + 16 + e + 2 g (rows g + 8).
template <bool KV8>
__device__ __forceinline__ int acc_dim(int mt, int r, int g) {
  if constexpr (KV8)
    return 32 * (mt >> 1) + (mt & 1) + 2 * g + ((r >> 1) << 4);
  else
    return mt * 16 + g + ((r >> 1) << 3);
}

// Byte offset of 16-byte chunk `chunk` (0 .. D/8-1) of tile row `row` in a
// TMA tile written with CU_TENSOR_MAP_SWIZZLE_128B: the chunk index inside a
// 128-byte row is XORed with (row mod 8).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * kBoxBytes + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

// Per-CTA bookkeeping shared by both decode kernels.
struct WorkItem {
  int b, hkv, h0, nh, split;
  int L, lo, nsplit;
  int u0, u1;  // virtual units of this CTA (see SeqUnits)
  SeqUnits su;
  bool len_ok, empty;
};

__device__ __forceinline__ WorkItem make_work_item(const DecodeParams& p) {
  WorkItem w;
  w.split = blockIdx.x;
  w.hkv = blockIdx.y / p.num_head_chunks;
  const int chunk = blockIdx.y - w.hkv * p.num_head_chunks;
  w.b = blockIdx.z;
  w.h0 = w.hkv * p.group + chunk * p.head_chunk;
  w.nh = min(p.head_chunk, p.group - chunk * p.head_chunk);
  w.L = p.context_lens[w.b];
  w.len_ok = w.L >= 0 && static_cast<int64_t>(w.L) <= static_cast<int64_t>(p.max_blocks) * p.block_size;
  w.su = seq_units(w.len_ok ? w.L : 0, p.window, p.num_sinks);
  w.lo = w.su.lo;
  w.empty = w.su.n_units == 0;
  w.nsplit = (!w.len_ok || w.empty) ? 1 : splits_for(w.su.n_units, p.units_per_split);
  w.u0 = w.split * p.units_per_split;
  w.u1 = min(w.u0 + p.units_per_split, w.su.n_units);
  return w;
}

// Rows of an invalid (NaN) or empty (zero) context, written by split 0.
template <typename T, int D>
__device__ void write_trivial_rows(const DecodeParams& p, const WorkItem& w) {
  const float val = w.len_ok ? 0.0f : __int_as_float(0x7fc00000);
  T* out = static_cast<T*>(p.out);
  for (int i = threadIdx.x; i < w.nh * D; i += blockDim.x) {
    const int qi = i / D, d = i - qi * D;
    out[(static_cast<int64_t>(w.b) * p.num_q_heads + w.h0 + qi) * D + d] = from_f32<T>(val);
  }
}

// Merge the per-warp softmax states held in shared memory and store either
// the final rows (single split) or this split's unnormalised partial.
//   so[w][q][DP] partial O, sm[w][q] running max (log2 units), sl[w][q] sum.
template <typename T, int D, int QT, int DP, int W = kDecodeWarps>
__device__ void merge_and_store(const float* so, const float* sm, const float* sl,
                                const DecodeParams& p, const WorkItem& w, bool bad) {
  const float nanf_ = __int_as_float(0x7fc00000);
  for (int i = threadIdx.x; i < w.nh * D; i += blockDim.x) {
    const int qi = i / D, d = i - qi * D;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < W; ++k) M = fmaxf(M, sm[k * QT + qi]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float mk = sm[k * QT + qi];
      const float f = (mk == -INFINITY) ? 0.f : ex2(mk - M);
      acc = fmaf(f, so[(k * QT + qi) * DP + d], acc);
      lsum = fmaf(f, sl[k * QT + qi], lsum);
    }
    const int64_t row = static_cast<int64_t>(w.b) * p.num_q_heads + (w.h0 + qi);
    if (w.nsplit == 1) {
      static_cast<T*>(p.out)[row * D + d] = from_f32<T>(bad ? nanf_ : acc / lsum);
    } else {
      const int64_t slot = row * p.num_splits + w.split;
      p.part_o[slot * D + d] = bad ? nanf_ : acc;
      if (d == 0) p.part_ml[slot] = make_float2(M, lsum);
    }
  }
}

// ---------------------------------------------------------------------------
// 16-bit pools: TMA-staged pages, tensor-core QK^T and PV.

template <typename T, int D, int NT, bool KV8, bool I8 = false, bool kShallow = false,
          int W = kDecodeWarps>
__global__ void __launch_bounds__(W * 32, W > kDecodeWarps ? 1
                                             : ((KV8 && NT == 1) ? 4 : (kShallow ? 3 : 2)))
decode16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const DecodeParams p) {
  using Cfg = Tile16<D, KV8, kShallow, W>;
  constexpr int QT = 8 * NT;        // query columns per CTA (padded group)
  constexpr int KS = D / 16;        // k-steps of QK^T == m-tiles of PV
  constexpr int DP = D + 4;         // padded row stride of the merge buffer
  constexpr int S = Cfg::kStages;
  static_assert(S <= 16, "the next chunk's pages are resolved 16 units ahead");
  static_assert(W * QT * (DP + 2) * 4 <= W * Cfg::kWarpBytes,
                "merge buffer must fit in the staging rings");
  static_assert(!KV8 || D == 128, "FP8 pools: head_dim 128");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[W][S];
  __shared__ int s_bad;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  pdl_wait_prior();
  const WorkItem w = make_work_item(p);
  if (!w.len_ok || w.empty) {
    if (w.split == 0) write_trivial_rows<T, D>(p, w);
    return;
  }
  if (w.split >= w.nsplit) return;

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;  // 128B-swizzle tiles need 1 KB alignment
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  const uint32_t ring = base_addr + warp * Cfg::kWarpBytes;
  const uint32_t scales = base_addr + W * Cfg::kWarpBytes + warp * Cfg::kScaleBytes;

  if (threadIdx.x == 0) s_bad = 0;
  if (lane == 0) {
    if (warp == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Units of this warp: u = u0 + warp + j * W.  Their pages are
  // resolved through the block table 32 at a time, lane l holding unit
  // 32 c + l of chunk c: y_cur holds the chunk of unit j, y_next the one
  // after it.  The next chunk's entries are read when a chunk starts and
  // examined only halfway through it, so the read never stalls the warp.
  const int span = w.u1 - w.u0;
  const int my_n = span > warp ? (span - warp + W - 1) / W : 0;
  auto unit_t0 = [&](int jj) -> int {  // first token of unit jj, -1 past the warp's units
    return jj < my_n ? phys_unit(w.su, w.u0 + warp + jj * W) * kUnitTokens : -1;
  };
  auto table_entry = [&](int t0) -> int32_t {
    return t0 < 0 ? -1
                  : __ldg(p.block_tables + static_cast<int64_t>(w.b) * p.max_blocks +
                          t0 / p.block_size);
  };
  // TMA row coordinate of the unit's first token, -1 = bad block id or no unit
  auto row_of = [&](int t0, int32_t pb) -> int {
    return (t0 >= 0 && pb >= 0 && pb < p.num_blocks)
               ? (pb * p.num_kv_heads + w.hkv) * p.block_size + (t0 % p.block_size)
               : -1;
  };
  int y_cur, y_next = -1;
  {
    const int t0 = unit_t0(lane);
    y_cur = row_of(t0, table_entry(t0));
  }
  int t0_ahead = unit_t0(32 + lane);  // the next chunk's entries, read ahead
  int32_t pb_ahead = table_entry(t0_ahead);
  // row coordinate of unit jj, jj in the current chunk or the next one
  auto y_of = [&](int jj, int j) -> int {
    const int v = (jj >> 5) == (j >> 5) ? y_cur : y_next;
    return __shfl_sync(0xffffffffu, v, jj & 31);
  };

  auto issue = [&](int stage, int y) {
    const uint32_t bar = smem_u32(&bars[warp][stage]);
    const uint32_t kdst = ring + stage * Cfg::kStageBytes;
    const uint32_t vdst = kdst + Cfg::kStageBytes / 2;
    if (y >= 0) {
      mbar_arrive_expect_tx(bar, Cfg::kTxBytes);
      if constexpr (KV8) {
        tma_load_2d(kdst, &kmap, 0, y, bar);  // 16 rows x 128 codes
        tma_load_2d(vdst, &vmap, 0, y, bar);
      } else if constexpr (D == 128) {
        // the 3-D view: both 64-column halves of the 16 rows in one copy
        tma_load_3d(kdst, &kmap, 0, y, 0, bar);
        tma_load_3d(vdst, &vmap, 0, y, 0, bar);
      } else {
        tma_load_2d(kdst, &kmap, 0, y, bar);
        tma_load_2d(vdst, &vmap, 0, y, bar);
      }
    } else {
      mbar_arrive(bar);  // nothing to fetch: complete the phase, the unit is flagged bad
    }
  };

  // 8-bit pools: the unit's 2 x 16 row scales come in by 4-byte cp.async
  // (lane l < 16: K row l, else V row l - 16), not as two more TMA copies:
  // each copy costs the SM's copy engine about as much to process as a whole
  // code tile.  Every lane commits one group per unit slot, empty when there
  // is nothing to fetch, so that the group of unit j is always the S-th
  // newest when unit j is read.
  auto issue_scales = [&](int stage, int y) {
    if constexpr (KV8) {
      if (y >= 0) {
        const float* src = (lane < kUnitTokens ? p.k_scale : p.v_scale) + y + (lane & (kUnitTokens - 1));
        cp_async_4(scales + stage * 2 * kUnitTokens * 4 + lane * 4, src);
      }
      cp_async_commit();
    }
  };

#pragma unroll
  for (int j = 0; j < S; ++j) {
    const int y = y_of(j, 0);
    if (lane == 0 && j < my_n) issue(j, y);
    issue_scales(j, j < my_n ? y : -1);
  }

  // Q fragments: B operand of S^T = K Q^T.  Lane holds q[n = lane/4] at
  // d = 16 kk + 2 (lane % 4) + {0, 1} (register 0) and + 8 (register 1).
  uint32_t qf[NT][KS][2];
  const int g = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi = nt * 8 + g;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(p.q) + (static_cast<int64_t>(w.b) * p.num_q_heads + w.h0 + qi) * D);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      if constexpr (KV8) {
        // the FP8 K fragments carry d = 16 kk + 4 tig + {0, 1} | + {2, 3}: match them
        const uint2 v2 = qi < w.nh ? __ldg(reinterpret_cast<const uint2*>(qrow + kk * 8) + tig)
                                   : make_uint2(0u, 0u);
        qf[nt][kk][0] = v2.x;
        qf[nt][kk][1] = v2.y;
      } else {
        qf[nt][kk][0] = qi < w.nh ? __ldg(qrow + kk * 8 + tig) : 0u;
        qf[nt][kk][1] = qi < w.nh ? __ldg(qrow + kk * 8 + 4 + tig) : 0u;
      }
    }
  }

  float o[KS][NT][4];
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      m_run[nt][jj] = -INFINITY;
      l_run[nt][jj] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) o[mt][nt][r] = 0.f;
  }
  bool bad = false;

  // Fused append: the warp that streams the unit holding position L-1 puts the
  // new token's K and V into that unit's staged rows -- so the token attends
  // to the new values -- and (head chunk 0 only) stores them to the pool slot.
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  const int t_new = w.L - 1;  // always inside the window part
  const int v_new = w.su.n_sink_u + t_new / kUnitTokens - w.su.win_u0;
  const int rel_new = v_new - w.u0 - warp;
  const bool own_new = p.k_new != nullptr && t_new >= 0 && rel_new >= 0 && v_new < w.u1 &&
                       rel_new % W == 0;
  const int j_new = own_new ? rel_new / W : -1;
  uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
  if (own_new && lane < 2 * CPR) {
    const T* src = static_cast<const T*>(lane < CPR ? p.k_new : p.v_new) +
                   (static_cast<int64_t>(w.b) * p.num_kv_heads + w.hkv) * D;
    new_row = __ldg(reinterpret_cast<const uint4*>(src) + (lane % CPR));
  }

  for (int j = 0; j < my_n; ++j) {
    if (my_n > 32) {  // (warp-uniform)
      if ((j & 31) == 16) y_next = row_of(t0_ahead, pb_ahead);  // read 16 units ago
      if ((j & 31) == 0 && j > 0) {
        y_cur = y_next;
        t0_ahead = unit_t0(j + 32 + lane);
        pb_ahead = table_entry(t0_ahead);
      }
    }
    const int stage = j % S;
    const uint32_t parity = (j / S) & 1;
    const int yj = y_of(j, j);
    const bool ok = mbar_wait_bounded(smem_u32(&bars[warp][stage]), parity, kWaitLimit);
    if (!__all_sync(0xffffffffu, ok)) {
      // The copy has not landed: stop using this ring.  Units j .. j+S-1 may
      // still have copies in flight, and the ring becomes the merge buffer
      // after the loop, so wait (bounded again) for each of them first.
      bad = true;
      for (int jj = j; jj < j + S && jj < my_n; ++jj)
        mbar_wait_bounded(smem_u32(&bars[warp][jj % S]), (jj / S) & 1, kWaitLimit);
      break;
    }
    if (yj < 0) bad = true;

    const uint32_t kt = ring + stage * Cfg::kStageBytes;
    const uint32_t vt = kt + Cfg::kStageBytes / 2;
    const int t0 = phys_unit(w.su, w.u0 + warp + j * W) * kUnitTokens;
    // per-row scales of the unit (FP8 pools; 1 otherwise): K rows g, g+8; V rows g, g+8
    float ksa = 1.f, ksb = 1.f, vsa = 1.f, vsb = 1.f;
    if constexpr (KV8) {
      cp_async_wait<S - 1>();  // this lane's scale copy of unit j has landed
      __syncwarp();            // ... and every other lane's
      const uint32_t sc = scales + stage * 2 * kUnitTokens * 4;
      ksa = ld_shared_f32(sc + (g << 2));
      ksb = ld_shared_f32(sc + ((g + 8) << 2));
      vsa = ld_shared_f32(sc + ((kUnitTokens + g) << 2));
      vsb = ld_shared_f32(sc + ((kUnitTokens + g + 8) << 2));
    }

    if (!KV8 && j == j_new) {
      const int r = t_new % kUnitTokens;
      if (lane < 2 * CPR) {
        const int c = lane % CPR;
        st_shared_v4((lane < CPR ? kt : vt) + swz(r, c), new_row);
        if (yj >= 0 && w.h0 == w.hkv * p.group) {
          T* dst = static_cast<T*>(lane < CPR ? p.k_dst : p.v_dst) +
                   (static_cast<int64_t>(yj) + r) * D;
          reinterpret_cast<uint4*>(dst)[c] = new_row;
        }
      }
      fence_proxy_async_smem();  // these generic writes precede the stage's next TMA fill
      __syncwarp();
    }

    // ---- S^T[16 tok x 8 NT q] = K[16 x D] . Q^T[D x 8 NT] ----
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) s[nt][r] = 0.f;
    if constexpr (KV8) {
      // one ldmatrix.x4 of codes = two k-steps of 16 d values for the 16 rows;
      // each 32-bit register holds 4 consecutive codes of one row
#pragma unroll
      for (int c = 0; c < KS / 2; ++c) {
        const int row = lane & 15, chunk = 2 * c + (lane >> 4);
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(kt + row * 128 + ((chunk ^ (row & 7)) << 4), r0, r1, r2, r3);
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        if constexpr (I8) {
          r0 ^= 0x80808080u;
          r1 ^= 0x80808080u;
          r2 ^= 0x80808080u;
          r3 ^= 0x80808080u;
          a0 = s8pair_to_f16x2<0x5140>(r0), a1 = s8pair_to_f16x2<0x5140>(r1);
          a2 = s8pair_to_f16x2<0x5342>(r0), a3 = s8pair_to_f16x2<0x5342>(r1);
          b0 = s8pair_to_f16x2<0x5140>(r2), b1 = s8pair_to_f16x2<0x5140>(r3);
          b2 = s8pair_to_f16x2<0x5342>(r2), b3 = s8pair_to_f16x2<0x5342>(r3);
        } else {
          a0 = e4m3x2_to_f16x2(r0), a1 = e4m3x2_to_f16x2(r1);
          a2 = e4m3x2_to_f16x2(r0 >> 16), a3 = e4m3x2_to_f16x2(r1 >> 16);
          b0 = e4m3x2_to_f16x2(r2), b1 = e4m3x2_to_f16x2(r3);
          b2 = e4m3x2_to_f16x2(r2 >> 16), b3 = e4m3x2_to_f16x2(r3 >> 16);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          Mma<T>::run(s[nt], a0, a1, a2, a3, qf[nt][2 * c][0], qf[nt][2 * c][1]);
          Mma<T>::run(s[nt], b0, b1, b2, b3, qf[nt][2 * c + 1][0], qf[nt][2 * c + 1][1]);
        }
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(kt + swz(lane & 15, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          Mma<T>::run(s[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
      }
    }

    // ---- scale into log2 units; mask tokens that are not attended ----
    const bool edge = !(t0 + kUnitTokens <= w.L &&
                        (t0 >= w.lo || t0 + kUnitTokens <= w.su.sinks));
    const int ta = t0 + g, tb = ta + 8;  // tokens of rows g and g + 8
    const bool va = !edge || attended(w.su, w.L, ta);
    const bool vb = !edge || attended(w.su, w.L, tb);
    const float fa = ksa * p.scale_log2, fb = ksb * p.scale_log2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      s[nt][0] = va ? s[nt][0] * fa : -INFINITY;
      s[nt][1] = va ? s[nt][1] * fa : -INFINITY;
      s[nt][2] = vb ? s[nt][2] * fb : -INFINITY;
      s[nt][3] = vb ? s[nt][3] * fb : -INFINITY;
    }

    // ---- column (query) maxima over the 16 tokens ----
    float mx[NT][2];
    bool need = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float v = fmaxf(s[nt][jj], s[nt][2 + jj]);
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        mx[nt][jj] = v;
        need |= v > m_run[nt][jj] + kRescaleThreshold;
      }
    // Lazy online softmax: move the reference max only when the new tile
    // exceeds it by more than the threshold (exact: every weight and the
    // accumulator share the reference).
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float mnew = mx[nt][jj] > m_run[nt][jj] + kRescaleThreshold ? mx[nt][jj] : m_run[nt][jj];
          const float alpha = ex2(m_run[nt][jj] - mnew);
          m_run[nt][jj] = mnew;
          l_run[nt][jj] *= alpha;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            o[mt][nt][jj] *= alpha;
            o[mt][nt][2 + jj] *= alpha;
          }
        }
    }

    // ---- weights P = 2^(s - m), split into hi + lo 16-bit parts, transposed ----
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float p0 = ex2(s[nt][0] - m_run[nt][0]);
      float p1 = ex2(s[nt][1] - m_run[nt][1]);
      float p2 = ex2(s[nt][2] - m_run[nt][0]);
      float p3 = ex2(s[nt][3] - m_run[nt][1]);
      l_run[nt][0] += p0 + p2;
      l_run[nt][1] += p1 + p3;
      if constexpr (KV8) {
        // fold the V row scales into the weights (masked rows have weight 0
        // and may carry a NaN scale)
        p0 = va ? p0 * vsa : 0.f;
        p1 = va ? p1 * vsa : 0.f;
        p2 = vb ? p2 * vsb : 0.f;
        p3 = vb ? p3 * vsb : 0.f;
      }
      const uint32_t htop = Mma<T>::pack(p0, p1), hbot = Mma<T>::pack(p2, p3);
      const uint32_t ltop = Mma<T>::pack(p0 - Mma<T>::lo_f32(htop), p1 - Mma<T>::hi_f32(htop));
      const uint32_t lbot = Mma<T>::pack(p2 - Mma<T>::lo_f32(hbot), p3 - Mma<T>::hi_f32(hbot));
      bh[nt][0] = movmatrix_trans(htop);
      bh[nt][1] = movmatrix_trans(hbot);
      bl[nt][0] = movmatrix_trans(ltop);
      bl[nt][1] = movmatrix_trans(lbot);
    }

    // ---- O^T[D x 8 NT] += V^T[D x 16] . P^T[16 x 8 NT] ----
    // Rows of V outside [lo, L) may hold anything (even NaN): zero them in
    // the fragment so that 0 * garbage cannot leak into the sum.
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (edge) {
      const int tk = t0 + 2 * tig;
      mlo = (attended(w.su, w.L, tk) ? 0x0000ffffu : 0u) |
            (attended(w.su, w.L, tk + 1) ? 0xffff0000u : 0u);
      mhi = (attended(w.su, w.L, tk + 8) ? 0x0000ffffu : 0u) |
            (attended(w.su, w.L, tk + 9) ? 0xffff0000u : 0u);
    }
    if constexpr (KV8) {
      // ldmatrix.trans on the code tile viewed as 16-bit pairs: a register
      // holds tokens (2 tig, 2 tig + 1) x dims (2 g, 2 g + 1) of one 16-d
      // chunk; one byte permute separates the even-d pair from the odd-d pair,
      // which feed the even and odd m-tiles of the 32-d block.  Units wholly
      // inside the context skip the masks (a second copy of the loop).
      auto v_products = [&](auto masked_tag) {
        constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
        for (int c = 0; c < KS / 2; ++c) {
          const int tok = (lane & 7) + ((lane >> 4) << 3);
          const int chunk = 2 * c + ((lane >> 3) & 1);
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(vt + tok * 128 + ((chunk ^ (tok & 7)) << 4), r0, r1, r2, r3);
          if constexpr (I8) {
            r0 ^= 0x80808080u;
            r1 ^= 0x80808080u;
            r2 ^= 0x80808080u;
            r3 ^= 0x80808080u;
          } else {
            r0 = __byte_perm(r0, 0u, 0x3120);
            r1 = __byte_perm(r1, 0u, 0x3120);
            r2 = __byte_perm(r2, 0u, 0x3120);
            r3 = __byte_perm(r3, 0u, 0x3120);
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t a0, a1, a2, a3;
            if constexpr (I8) {  // even d: bytes 0, 2; odd d: bytes 1, 3
              a0 = e ? s8pair_to_f16x2<0x5341>(r0) : s8pair_to_f16x2<0x5240>(r0);
              a1 = e ? s8pair_to_f16x2<0x5341>(r1) : s8pair_to_f16x2<0x5240>(r1);
              a2 = e ? s8pair_to_f16x2<0x5341>(r2) : s8pair_to_f16x2<0x5240>(r2);
              a3 = e ? s8pair_to_f16x2<0x5341>(r3) : s8pair_to_f16x2<0x5240>(r3);
            } else {
              const int sh = 16 * e;
              a0 = e4m3x2_to_f16x2(r0 >> sh);
              a1 = e4m3x2_to_f16x2(r1 >> sh);
              a2 = e4m3x2_to_f16x2(r2 >> sh);
              a3 = e4m3x2_to_f16x2(r3 >> sh);
            }
            if constexpr (kMasked) {
              a0 &= mlo;
              a1 &= mlo;
              a2 &= mhi;
              a3 &= mhi;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              Mma<T>::run(o[2 * c + e][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
              Mma<T>::run(o[2 * c + e][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
            }
          }
        }
      };
      if (edge) {
        v_products(std::true_type{});
      } else {
        v_products(std::false_type{});
      }
    } else {
      auto v_products = [&](auto masked_tag) {
        constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t a0, a1, a2, a3;
          const int tok = (lane & 7) + ((lane >> 4) << 3);
          ldmatrix_x4_trans(vt + swz(tok, mt * 2 + ((lane >> 3) & 1)), a0, a1, a2, a3);
          if constexpr (kMasked) {
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            Mma<T>::run(o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
            Mma<T>::run(o[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
          }
        }
      };
      if (edge) {
        v_products(std::true_type{});
      } else {
        v_products(std::false_type{});
      }
    }

    // ---- recycle the stage ----
    fence_proxy_async_smem();  // this lane's reads of the stage precede the refill
    __syncwarp();
    const int yn = j + S < my_n ? y_of(j + S, j) : -1;
    if (lane == 0 && j + S < my_n) issue(stage, yn);
    issue_scales(stage, yn);
  }
  if constexpr (KV8) cp_async_wait<0>();  // no copy into shared memory outlives the loop

  // ---- per-warp state -> shared memory -> CTA merge ----
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      float v = l_run[nt][jj];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[nt][jj] = v;
    }
  if (bad) s_bad = 1;
  __syncthreads();  // every warp is done with its ring; reuse it for the merge

  float* so = reinterpret_cast<float*>(base);
  float* sm = so + W * QT * DP;
  float* sl = sm + W * QT;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = acc_dim<KV8>(mt, r, g);
        const int q = nt * 8 + 2 * tig + (r & 1);
        so[(warp * QT + q) * DP + d] = o[mt][nt][r];
      }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        sm[warp * QT + nt * 8 + 2 * tig + jj] = m_run[nt][jj];
        sl[warp * QT + nt * 8 + 2 * tig + jj] = l_run[nt][jj];
      }
  }
  __syncthreads();
  merge_and_store<T, D, QT, DP, W>(so, sm, sl, p, w, s_bad != 0);
}

// ---------------------------------------------------------------------------
// fp32 pools: CUDA-core path with the same work split.

// fp32 pools: warps per CTA (each a unit at a time; short contexts need
// more of them side by side to hide the memory latency)
constexpr int kF32Warps = 8;

// QT: query heads a CTA computes (1, 2, 4 or 8: the plan's head chunk
// rounded up), so that an MHA pool does no work for seven empty heads.
template <int D, int QT>
__global__ void __launch_bounds__(kF32Warps * 32)
decode_f32_kernel(const DecodeParams p) {
  constexpr int LPR = D / 4;     // lanes per context row (one float4 each)
  constexpr int RPW = 32 / LPR;  // rows per warp step
  constexpr int DP = D + 4;
  __shared__ float so[kF32Warps * QT * DP];
  __shared__ float sm[kF32Warps * QT];
  __shared__ float sl[kF32Warps * QT];
  __shared__ int s_bad;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  pdl_wait_prior();
  const WorkItem w = make_work_item(p);
  if (!w.len_ok || w.empty) {
    if (w.split == 0) write_trivial_rows<float, D>(p, w);
    return;
  }
  if (w.split >= w.nsplit) return;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();

  const int sub = lane / LPR;  // which row of the warp step
  const int li = lane % LPR;   // float4 column
  float4 qv[QT];
#pragma unroll
  for (int qi = 0; qi < QT; ++qi) {
    qv[qi] = qi < w.nh
                 ? __ldg(reinterpret_cast<const float4*>(
                             static_cast<const float*>(p.q) +
                             (static_cast<int64_t>(w.b) * p.num_q_heads + w.h0 + qi) * D) + li)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m[QT], l[QT];
  float4 acc[QT];
#pragma unroll
  for (int qi = 0; qi < QT; ++qi) {
    m[qi] = -INFINITY;
    l[qi] = 0.f;
    acc[qi] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  bool bad = false;
  const float* kc = static_cast<const float*>(p.k_cache);
  const float* vc = static_cast<const float*>(p.v_cache);

  // Rows of a unit come in batches of kBatch warp steps, all their loads
  // issued before any of them is used (one round trip to memory per batch,
  // not per row); the next unit's block-table entry is read while the
  // current unit's rows are in flight.
  constexpr int kSteps = kUnitTokens / RPW;
  constexpr int kBatch = D == 128 ? 4 : (kSteps < 8 ? kSteps : 8);  // (D 128: no spills)
  auto page_of = [&](int u) -> int32_t {
    return u < w.u1 ? __ldg(p.block_tables + static_cast<int64_t>(w.b) * p.max_blocks +
                            phys_unit(w.su, u) * kUnitTokens / p.block_size)
                    : -1;
  };
  int32_t pb_next = page_of(w.u0 + warp);
  for (int u = w.u0 + warp; u < w.u1; u += kF32Warps) {
    const int t0 = phys_unit(w.su, u) * kUnitTokens;
    const int32_t pb = pb_next;
    pb_next = page_of(u + kF32Warps);
    if (pb < 0 || pb >= p.num_blocks) {
      bad = true;
      continue;
    }
    const int64_t tile = ((static_cast<int64_t>(pb) * p.num_kv_heads + w.hkv) * p.block_size +
                          (t0 % p.block_size)) * D;
    for (int s0 = 0; s0 < kSteps; s0 += kBatch) {
      float4 kb[kBatch], vb[kBatch];
      bool vok[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int r = sub + (s0 + i) * RPW;
        const int t = t0 + r;
        const bool valid = attended(w.su, w.L, t);
        vok[i] = valid;
        kb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        vb[i] = kb[i];
        if (valid && p.k_new != nullptr && t == w.L - 1) {
          // fused append: attend to the new token and store it to its slot
          const int64_t src = (static_cast<int64_t>(w.b) * p.num_kv_heads + w.hkv) * D;
          kb[i] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.k_new) + src) + li);
          vb[i] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.v_new) + src) + li);
          if (w.h0 == w.hkv * p.group) {
            reinterpret_cast<float4*>(static_cast<float*>(p.k_dst) + tile + r * D)[li] = kb[i];
            reinterpret_cast<float4*>(static_cast<float*>(p.v_dst) + tile + r * D)[li] = vb[i];
          }
        } else if (valid) {
          kb[i] = __ldg(reinterpret_cast<const float4*>(kc + tile + r * D) + li);
          vb[i] = __ldg(reinterpret_cast<const float4*>(vc + tile + r * D) + li);
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const bool valid = vok[i];
        const float4 k4 = kb[i], v4 = vb[i];
#pragma unroll
        for (int qi = 0; qi < QT; ++qi) {
          float part = qv[qi].x * k4.x + qv[qi].y * k4.y + qv[qi].z * k4.z + qv[qi].w * k4.w;
#pragma unroll
          for (int off = 1; off < LPR; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
          if (valid) {
            const float sc = part * p.scale_log2;
            const float mnew = fmaxf(m[qi], sc);
            const float alpha = ex2(m[qi] - mnew);
            const float pw = ex2(sc - mnew);
            m[qi] = mnew;
            l[qi] = l[qi] * alpha + pw;
            acc[qi].x = acc[qi].x * alpha + pw * v4.x;
            acc[qi].y = acc[qi].y * alpha + pw * v4.y;
            acc[qi].z = acc[qi].z * alpha + pw * v4.z;
            acc[qi].w = acc[qi].w * alpha + pw * v4.w;
          }
        }
      }
    }
  }
  // merge the row groups of the warp (RPW == 2 for D == 64)
  if (RPW == 2) {
#pragma unroll
    for (int qi = 0; qi < QT; ++qi) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[qi], 16);
      const float lo_ = __shfl_xor_sync(0xffffffffu, l[qi], 16);
      float4 ao;
      ao.x = __shfl_xor_sync(0xffffffffu, acc[qi].x, 16);
      ao.y = __shfl_xor_sync(0xffffffffu, acc[qi].y, 16);
      ao.z = __shfl_xor_sync(0xffffffffu, acc[qi].z, 16);
      ao.w = __shfl_xor_sync(0xffffffffu, acc[qi].w, 16);
      const float M = fmaxf(m[qi], mo);
      const float fa = m[qi] == -INFINITY ? 0.f : ex2(m[qi] - M);
      const float fb = mo == -INFINITY ? 0.f : ex2(mo - M);
      m[qi] = M;
      l[qi] = l[qi] * fa + lo_ * fb;
      acc[qi].x = acc[qi].x * fa + ao.x * fb;
      acc[qi].y = acc[qi].y * fa + ao.y * fb;
      acc[qi].z = acc[qi].z * fa + ao.z * fb;
      acc[qi].w = acc[qi].w * fa + ao.w * fb;
    }
  }
  if (bad) s_bad = 1;
  if (sub == 0) {
#pragma unroll
    for (int qi = 0; qi < QT; ++qi) {
      float* dst = so + (warp * QT + qi) * DP + li * 4;
      dst[0] = acc[qi].x;
      dst[1] = acc[qi].y;
      dst[2] = acc[qi].z;
      dst[3] = acc[qi].w;
      if (li == 0) {
        sm[warp * QT + qi] = m[qi];
        sl[warp * QT + qi] = l[qi];
      }
    }
  }
  __syncthreads();
  merge_and_store<float, D, QT, DP, kF32Warps>(so, sm, sl, p, w, s_bad != 0);
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine of the split partials: one warp per (sequence, head).
//   M = max_s m_s,  out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.

template <typename T, int D>
__global__ void __launch_bounds__(128)
combine_kernel(const DecodeParams p) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  pdl_wait_prior();
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (item >= static_cast<int64_t>(p.num_seqs) * p.num_q_heads) return;
  const int b = static_cast<int>(item / p.num_q_heads);
  const int L = p.context_lens[b];
  if (L < 0 || static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks) * p.block_size) return;
  const int nsplit = splits_for(seq_units(L, p.window, p.num_sinks).n_units, p.units_per_split);
  if (nsplit <= 1) return;  // written directly by the decode kernel

  const float2* ml = p.part_ml + item * p.num_splits;
  const float* po = p.part_o + item * p.num_splits * D;
  float M = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, ml[s].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float2 v = ml[s];
    const float f = v.x == -INFINITY ? 0.f : ex2(v.x - M);
    lsum = fmaf(f, v.y, lsum);
    const float* src = po + static_cast<int64_t>(s) * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = fmaf(f, src[i], acc[i]);
  }
  T* out = static_cast<T*>(p.out) + item * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; ++i) out[i] = from_f32<T>(acc[i] / lsum);
}

template <typename T, int D, int NT, bool KV8 = false, bool I8 = false, bool kShallow = false,
          int W = kDecodeWarps>
cudaError_t launch16(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                     cudaStream_t stream) {
  auto kern = decode16_kernel<T, D, NT, KV8, I8, kShallow, W>;
  const int smem = Tile16<D, KV8, kShallow, W>::kSmemBytes;
  // the shared-memory opt-in is per device; set it once for each
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  dim3 grid(p.num_splits, p.num_kv_heads * p.num_head_chunks, p.num_seqs);
  return launch_pdl(kern, grid, dim3(W * 32), smem, stream, kmap, vmap, p);
}

}  // namespace

cudaError_t launch_decode_q8(bool int8, int ntiles, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, const DecodeParams& p, cudaStream_t stream) {
  if (int8) {
    if (ntiles == 1) return launch16<__half, 128, 1, true, true>(kmap, vmap, p, stream);
    return launch16<__half, 128, 2, true, true>(kmap, vmap, p, stream);
  }
  if (ntiles == 1) return launch16<__half, 128, 1, true>(kmap, vmap, p, stream);
  return launch16<__half, 128, 2, true>(kmap, vmap, p, stream);
}

cudaError_t launch_decode_16bit(int dtype, int head_dim, int ntiles, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const DecodeParams& p,
                                cudaStream_t stream) {
  // Many short work items (a serving batch: 54 per SM): two ring stages and
  // three CTAs per SM hide more of each item's start-up (+18 % on the serving
  // mix); fewer, longer ones keep three stages (a long sliding window: two
  // stages measured 3 % slower; the long MHA / GQA batches, 13 items per SM:
  // 0.3 % slower).
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const int64_t items = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * p.num_head_chunks;
  const bool shallow = head_dim == 128 && ntiles == 1 && items >= 16 * static_cast<int64_t>(sms);
  // A grid of at most one CTA per SM (a window per item, one split each):
  // twelve warps of two ring stages per CTA, so that each SM runs more than
  // four warps' chains (eight warps of three stages: 1.8 % slower).
  const bool wide = head_dim == 128 && ntiles == 1 &&
                    items * p.num_splits <= static_cast<int64_t>(sms);
  // dtype: 1 = fp16, 2 = bf16
#define PKV_LAUNCH16(T, D, NT) return launch16<T, D, NT>(kmap, vmap, p, stream)
  if (dtype == 1) {
    if (head_dim == 128) {
      if (ntiles == 1 && shallow) return launch16<__half, 128, 1, false, false, true>(kmap, vmap, p, stream);
      if (wide) return launch16<__half, 128, 1, false, false, true, 12>(kmap, vmap, p, stream);
      if (ntiles == 1) PKV_LAUNCH16(__half, 128, 1);
      PKV_LAUNCH16(__half, 128, 2);
    }
    if (ntiles == 1) PKV_LAUNCH16(__half, 64, 1);
    PKV_LAUNCH16(__half, 64, 2);
  }
  if (head_dim == 128) {
    if (ntiles == 1 && shallow)
      return launch16<__nv_bfloat16, 128, 1, false, false, true>(kmap, vmap, p, stream);
    if (wide) return launch16<__nv_bfloat16, 128, 1, false, false, true, 12>(kmap, vmap, p, stream);
    if (ntiles == 1) PKV_LAUNCH16(__nv_bfloat16, 128, 1);
    PKV_LAUNCH16(__nv_bfloat16, 128, 2);
  }
  if (ntiles == 1) PKV_LAUNCH16(__nv_bfloat16, 64, 1);
  PKV_LAUNCH16(__nv_bfloat16, 64, 2);
#undef PKV_LAUNCH16
}

template <int D>
cudaError_t launch_f32_d(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  const dim3 block(kF32Warps * 32);
  if (p.head_chunk <= 1) return launch_pdl(decode_f32_kernel<D, 1>, grid, block, 0, stream, p);
  if (p.head_chunk <= 2) return launch_pdl(decode_f32_kernel<D, 2>, grid, block, 0, stream, p);
  if (p.head_chunk <= 4) return launch_pdl(decode_f32_kernel<D, 4>, grid, block, 0, stream, p);
  return launch_pdl(decode_f32_kernel<D, 8>, grid, block, 0, stream, p);
}

cudaError_t launch_decode_f32(int head_dim, const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.num_splits, p.num_kv_heads * p.num_head_chunks, p.num_seqs);
  if (p.head_chunk > 8) return cudaErrorInvalidConfiguration;  // the plan caps fp32 at 8
  if (head_dim == 128) return launch_f32_d<128>(p, grid, stream);
  return launch_f32_d<64>(p, grid, stream);
}

cudaError_t launch_combine(int dtype, int head_dim, const DecodeParams& p, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
  if (items == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((items + 3) / 4);
#define PKV_COMBINE(T, D) \
  return launch_pdl(combine_kernel<T, D>, dim3(blocks), dim3(128), 0, stream, p)
  if (dtype == 0) {
    if (head_dim == 128) PKV_COMBINE(float, 128);
    PKV_COMBINE(float, 64);
  }
  if (dtype == 1) {
    if (head_dim == 128) PKV_COMBINE(__half, 128);
    PKV_COMBINE(__half, 64);
  }
  if (head_dim == 128) PKV_COMBINE(__nv_bfloat16, 128);
  PKV_COMBINE(__nv_bfloat16, 64);
#undef PKV_COMBINE
}

}  // namespace pkv
