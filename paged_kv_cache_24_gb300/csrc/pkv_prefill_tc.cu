// pkv_prefill_tc.cu -- chunked prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators and probabilities in tensor memory).
//
// What is computed: see pkv_prefill.cu ("Building a Streaming Sliding-Window
// Attention Engine in Pure Python", Step 3, prefill_attention: the query at
// position p attends keys j <= p with p - j < window, softmax per row; with
// a window, the first num_sinks positions too -- the attention sinks of that
// page's Extending list).
//
// How.  A CTA owns 256 query rows of one (sequence, kv head): (token, GQA
// head) pairs, so every K/V page it reads serves the whole group.  CTAs take
// the (sequence, token chunk) items in the order the planner gave them
// (most key tiles first), the kv heads of one item side by side.  The rows
// form two tiles of 128 (one per TMEM lane), worked on in ping-pong over
// tiles of 128 keys (with sinks: the sink tiles first, then the window's):
//   warp 9       (load)    TMA of the 16-key K and V units of each key tile
//                          into two rings of stages (128-byte swizzle), lane
//                          i issuing unit i's copies;
//   warps 10-11  (V prep)  turn each landed V tile into fp16 in place (bf16
//                          caches) and zero the rows of keys no row of the CTA
//                          may see, so garbage (even NaN) in unused slots
//                          cannot leak through a zero weight;
//   warp 8       (MMA)     one thread waits and issues S_t = Q_t K^T (M 128, N 128, both
//                          operands K-major in shared memory) and
//                          O_t += P_t V (A = P_t read from TMEM, B = V read
//                          MN-major from its stage);
//   warps 0-3 / 4-7        tile 0 / tile 1 softmax: each thread owns one row
//                          (its TMEM lane), loads its 128 scores, masks, keeps
//                          the running maximum and sum, writes P as fp16 over
//                          the scores it came from, and, when the maximum
//                          moved by more than 2^8, rescales its O row in TMEM
//                          (lazy rescaling).
// bf16 caches: the P.V product runs in fp16 on V scaled by a power of two
// 2^k chosen per (sequence, kv head) from the range of its V values (found by
// the append launch before this one), so that every scaled value is exactly
// an fp16 value; the output is scaled back by 2^-k.  A (sequence, kv head)
// whose values span more than fp16 can hold exactly, or that holds an
// infinity or NaN, is left to a second launch of this kernel (kExact): V
// stays bf16 and P comes as a hi + lo pair of bf16 parts (two P.V
// products), exact over bf16's whole range.
// While one tile's rows are in the softmax, the tensor cores work on the
// other tile's products.  The softmax warpgroups take registers from the
// others (setmaxnreg).
#include <atomic>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_prefill.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kQT = 128;          // rows per Q tile == TMEM lanes
constexpr int kRowsCta = kPrefillRowsCta;
constexpr int kTKeys = kPrefillTileKeys;  // keys per K/V tile
static_assert(kRowsCta == 2 * kQT && kUnitTokens == 16, "tile shapes");
constexpr int kTUnits = kTKeys / kUnitTokens;
constexpr int kMmaWarp = 8, kLoadWarp = 9, kPrepWarp0 = 10;
constexpr int kTThreads = 384;
constexpr int kPrepThreads = kTThreads - kPrepWarp0 * 32;
constexpr float kTRescale = 8.0f;
// register split: the two softmax warpgroups grow, the third shrinks; the sum
// must not exceed what the block is launched with (checked on the host)
constexpr int kSoftmaxRegs = 200, kOtherRegs = 104;

struct TcParams {
  const void* q;
  void* out;
  const int32_t* cu_q;
  const int32_t* order;  // work items, most key tiles first
  const int32_t* block_tables;
  const int32_t* context_lens;
  int64_t num_blocks;
  int num_q_heads, num_kv_heads, group;
  int head_chunk_log2, num_head_chunks, chunks_per_seq;
  int num_sinks;  // attention sinks (0 without a window)
  int max_blocks, block_size, window;
  float scale_log2;
  // bf16 caches: per (sequence, kv head), row_blocks partial ranges of its V
  // magnitudes (largest, smallest non-zero minus one; bf16 bits), and per
  // CTA the first launch's choice for the second (0: done, else 1 + down_c)
  const uint2* vparts;
  int row_blocks;
  uint32_t* mode;
};

template <int D>
struct TcLayout {
  static constexpr int kKStages = D == 128 ? 2 : 3;  // stages per ring
  static constexpr int kVStages = kKStages;
  static constexpr int kKBlocks = D / 64;                   // 128-byte column blocks
  static constexpr int kQTileBytes = kKBlocks * kQT * 128;
  static constexpr int kKVTile = kKBlocks * kTKeys * 128;   // K (or V) of one key tile
  // V tiles are unit-major: unit u (16 keys) at u * kVUnitBytes, its 64-column
  // blocks 2 KB apart, so one 3-D copy brings a unit's rows (K tiles keep
  // each 64-column block of all 128 keys together, as the S product needs)
  static constexpr int kVUnitBytes = kKBlocks * kUnitTokens * 128;
  static constexpr int kKOff = 2 * kQTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kKVTile;
  static constexpr int kSmemBytes = kVOff + kVStages * kKVTile;
  // TMEM columns: O_t at t*D, S_t (and P_t over its first 64) at 2D + 128t
  static constexpr uint32_t o_col(int t) { return static_cast<uint32_t>(t * D); }
  static constexpr uint32_t s_col(int t) { return static_cast<uint32_t>(2 * D + 128 * t); }
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * D + 256 <= 512, "TMEM columns");
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// two bf16 (low half first) times a power of two -> two fp16, rounded to
// nearest: exact when the scaled values are fp16 values (see VRange)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float2 up) {
  const float2 x = __fmul2_rn(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)),
                              up);
  return Mma<__half>::pack(x.x, x.y);
}

// What the V range of a (sequence, kv head) allows.  mx: the largest
// magnitude of its bf16 V values (as bits), mn1: the smallest non-zero one
// minus one (as bits).
//   up:     2^k, k in [-126, 126], putting the largest magnitude in [2^14, 2^15);
//   exact:  some value would not be exactly an fp16 value after the scaling
//           (below 2^-17 its last significant bit falls under fp16's
//           subnormal step 2^-24), or the range holds an infinity or NaN:
//           the kExact launch takes the pair;
//   down_c: kExact only, weights scaled by 2^-down_c so that P.V sums of
//           values near bf16's top stay inside fp32's range.
struct VRange {
  float up, down;
  int down_c;
  bool exact;
};
__device__ __forceinline__ VRange v_range_decision(uint32_t mx, uint32_t mn1) {
  VRange r{1.f, 1.f, 0, false};
  if (mx == 0u) return r;  // all zero
  if (mx >= 0x7f80u) {     // an infinity or NaN
    r.exact = true;
    return r;
  }
  const int e = static_cast<int>(mx >> 7);  // biased exponent of the largest value
  const int k = max(-126, min(126, 141 - max(e, 1)));
  r.up = __int_as_float((127 + k) << 23);
  r.down = __int_as_float((127 - k) << 23);
  const float hi = __uint_as_float(mx << 16) * r.up;
  const float lo = __uint_as_float((mn1 + 1u) << 16) * r.up;
  if (!(hi <= 65280.f && lo >= 0x1p-17f)) {
    // V stays as it is in the kExact launch
    r.exact = true;
    r.up = r.down = 1.f;
    r.down_c = max(0, e - 227);  // 2^100 and above
  }
  return r;
}

// Two probabilities as a hi + lo pair of bf16 values (low half first in each
// word): hi = p rounded to bf16, lo = the remainder p - hi (exact in fp32)
// rounded to bf16, so hi + lo carries p to about 2^-17 of itself over bf16's
// range (a single bf16 P would lose up to 2^-9 of each weight).
__device__ __forceinline__ void split_bf16x2(float2 pr, uint32_t& hi, uint32_t& lo) {
  hi = Mma<__nv_bfloat16>::pack(pr.x, pr.y);
  const float2 hf = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u));
  const float2 r = ffma2(hf, make_float2(-1.f, -1.f), pr);
  lo = Mma<__nv_bfloat16>::pack(r.x, r.y);
}

// kSinks: the key range has a sink section (window > 0, num_sinks > 0); the
// instantiation without it compiles the sink tests away.  kExact (bf16
// caches): the second launch -- only the CTAs of (sequence, kv head) pairs
// whose V range fp16 cannot hold run, with V in bf16 and P as hi + lo bf16
// parts.
template <typename T, int D, bool kSinks, bool kExact>
__global__ void __launch_bounds__(kTThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const TcParams p) {
  using Lay = TcLayout<D>;
  constexpr int SK = Lay::kKStages, SV = Lay::kVStages;
  constexpr bool kBf16 = __is_same(T, __nv_bfloat16);
  static_assert(!kExact || kBf16, "the kExact launch is for bf16 caches");
  constexpr bool kConvert = kBf16 && !kExact;  // V to fp16 (scaled) in shared memory
  constexpr uint32_t kIdS = umma_idesc_f16(kBf16 ? 1u : 0u, kQT, kTKeys, 0);
  // P.V: P and V in fp16, or (kExact) both in bf16
  constexpr uint32_t kIdO = umma_idesc_f16(kExact ? 1u : 0u, kQT, D, 1);

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[SK], k_empty[SK], v_full[SV], v_ready[SV], v_empty[SV];
  __shared__ __align__(8) uint64_t s_full[2], p_full[2], o_done[2], done_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int s_bad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  pdl_wait_prior();
  VRange vr{1.f, 1.f, 0, false};
  if constexpr (kExact) {
    const uint32_t m = p.mode[blockIdx.x];  // the first launch's choice
    if (m == 0u) return;
    vr = VRange{1.f, 1.f, static_cast<int>(m) - 1, true};
  }

  const int hh_count = p.num_kv_heads * p.num_head_chunks;
  const int slot = static_cast<int>(blockIdx.x / hh_count);
  const int hh = static_cast<int>(blockIdx.x - static_cast<unsigned>(slot) * hh_count);
  const int item = p.order[slot];
  const int b = item / p.chunks_per_seq;
  const int hkv = hh / p.num_head_chunks;
  const int chunk = hh - hkv * p.num_head_chunks;
  const int lg = p.head_chunk_log2, gc = 1 << lg;
  const int tok_per_cta = kRowsCta >> lg;
  // bf16 caches: the pair's partial V ranges (at most two per lane), read
  // alongside the work item's own loads
  static_assert(kPrefillScanParts <= 64, "two partials per lane");
  uint2 part_r[2] = {make_uint2(0u, 0xffffffffu), make_uint2(0u, 0xffffffffu)};
  if constexpr (kConvert) {
    const uint2* part = p.vparts + (static_cast<int64_t>(b) * p.num_kv_heads + hkv) * p.row_blocks;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (lane + 32 * q < p.row_blocks) part_r[q] = __ldg(part + lane + 32 * q);
  }
  const PrefillItem it = prefill_item(p.cu_q, p.context_lens, b, item - b * p.chunks_per_seq,
                                      tok_per_cta, p.window, p.num_sinks, p.max_blocks,
                                      p.block_size);
  if (it.empty) {
    if (kConvert && tid == 0) p.mode[blockIdx.x] = 0u;
    return;
  }
  if constexpr (kConvert) {
    // bf16 caches: this launch takes the pairs whose V range scales into fp16
    // exactly and leaves the others to the kExact launch (each warp reduces
    // the pair's partial ranges itself)
    const uint32_t mx = max(part_r[0].x, part_r[1].x), mn = min(part_r[0].y, part_r[1].y);
    vr = v_range_decision(__reduce_max_sync(0xffffffffu, mx), __reduce_min_sync(0xffffffffu, mn));
    if (tid == 0) p.mode[blockIdx.x] = vr.exact ? 1u + static_cast<uint32_t>(vr.down_c) : 0u;
    if (vr.exact) return;
  }
  const int start = it.start, tile0 = it.tile0, tile_n = it.tile_n;
  const int pos0 = it.pos0, pos1 = it.pos1, k_lo = it.k_lo;
  const int n_units = it.n_units, n_tiles = it.n_tiles;
  const int sink_tiles = kSinks ? it.sink_tiles : 0, sink_units = kSinks ? it.sink_units : 0;
  const int win_u0 = it.win_u0;
  const int sink_end = sink_units * kUnitTokens;  // keys of the sink section
  const int num_sinks = kSinks ? p.num_sinks : 0;
  const bool len_ok = it.len_ok;
  // first key position of key tile j (the sink tiles, then the window tiles)
  auto tile_t0 = [&](int j) {
    return j < sink_tiles ? j * kTKeys : (win_u0 + (j - sink_tiles) * kTUnits) * kUnitTokens;
  };
  // keys some row of the CTA attends and tile j holds: at most pos1, inside the
  // window of some row or a sink, and (sink tiles) inside the sink section
  auto key_kept = [&](int j, int kp) {
    return kp <= pos1 && (j >= sink_tiles || kp < sink_end) &&
           (p.window <= 0 || kp >= k_lo || kp < num_sinks);
  };

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;

  // ---- set-up: TMEM, barriers, the Q tiles ----
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(Lay::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == kMmaWarp * 32) {
    for (int s = 0; s < SK; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_ready[s]), kPrepThreads);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&s_full[t]), 1);
      mbar_init(smem_u32(&p_full[t]), kQT);
      mbar_init(smem_u32(&o_done[t]), 1);
    }
    mbar_init(smem_u32(&done_bar), 1);
    s_bad = len_ok ? 0 : 1;
    fence_mbar_init();
  }
  // softmax threads: row `row` of Q tile `wg` (token ti of the CTA, head hi of the chunk)
  const int wg = warp >> 2, row = tid & (kQT - 1);
  const int r_cta = wg * kQT + row;
  const int ti = r_cta >> lg, hi = r_cta & (gc - 1);
  const bool row_ok = warp < 8 && ti < tile_n;
  const int rpos = row_ok ? pos0 + ti : -1;
  const int64_t qo_row = (static_cast<int64_t>(start + tile0 + (row_ok ? ti : 0)) * p.num_q_heads +
                          hkv * p.group + chunk * gc + hi) * D;
  if (warp < 8) {
    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + qo_row);
    const uint32_t qt = base + wg * Lay::kQTileBytes;
#pragma unroll
    for (int c16 = 0; c16 < D / 8; ++c16) {
      const uint4 v = row_ok ? __ldg(qrow + c16) : make_uint4(0u, 0u, 0u, 0u);
      st_shared_v4(qt + (c16 >> 3) * kQT * 128 + sw128(row, c16), v);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  bool bad = false;
  auto k_addr = [&](int j) { return base + Lay::kKOff + (j % SK) * Lay::kKVTile; };
  auto v_addr = [&](int j) { return base + Lay::kVOff + (j % SV) * Lay::kKVTile; };

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kLoadWarp) {
      // ============ load warp: K and V units of each key tile into their rings ============
      if (lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
      }
      // First key position of virtual unit u (the sink tiles' units, then the
      // window's), -1 past the range or in the sink tiles' padding.
      auto unit_t0 = [&](int u) -> int {
        if (u >= n_units) return -1;
        if constexpr (kSinks) {
          const int su = sink_tiles * kTUnits;
          if (u < su && u >= sink_units) return -1;
          return (u < su ? u : win_u0 + (u - su)) * kUnitTokens;
        } else {
          return (win_u0 + u) * kUnitTokens;
        }
      };
      auto table_entry = [&](int t0) -> int32_t {
        return __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks + t0 / p.block_size);
      };
      // page row of the unit at t0 with block id pb: -1 past the range, -2 invalid page
      auto page_y = [&](int t0, int32_t pb) -> int {
        if (t0 < 0) return -1;
        if (pb < 0 || pb >= p.num_blocks) return -2;
        return (pb * p.num_kv_heads + hkv) * p.block_size + (t0 % p.block_size);
      };
      // Lane 0 posts the tile's byte count, then lane i copies unit i (its
      // K rows one box per 64 columns, its V rows in one box): a copy takes
      // tens of cycles to issue, so the eight units go out side by side.
      auto issue = [&](const CUtensorMap* map, uint32_t bar, uint32_t dst, int y, int loaded,
                       bool v_tile) {
        if (lane == 0) {
          if (loaded == 0)
            mbar_arrive(bar);
          else
            mbar_arrive_expect_tx(bar, loaded * Lay::kKBlocks * kUnitTokens * 128);
        }
        __syncwarp();
        if (y >= 0) {
          if (v_tile) {
            // the V map of a 128-column pool is 3-D: both column blocks of the
            // unit's 16 rows in one box
            if constexpr (D == 128)
              tma_load_3d(dst + lane * Lay::kVUnitBytes, map, 0, y, 0, bar);
            else
              tma_load_2d(dst + lane * Lay::kVUnitBytes, map, 0, y, bar);
          } else {
#pragma unroll
            for (int kb = 0; kb < Lay::kKBlocks; ++kb)
              tma_load_2d(dst + kb * kTKeys * 128 + lane * kUnitTokens * 128, map, kb * 64, y,
                          bar);
          }
        }
      };
      // lane i < 8 holds the page row of unit i of the tile (-1 elsewhere)
      int y_next = -1;
      if (lane < kTUnits && n_tiles > 0) {
        const int t0 = unit_t0(lane);
        y_next = page_y(t0, t0 >= 0 ? table_entry(t0) : -1);
      }
      for (int j = 0; j < n_tiles; ++j) {
        const int y_cur = y_next;
        // the next tile's block-table entries: read now, examined only after
        // this tile's copies are out, so the read's latency overlaps them
        const int t0n = (lane < kTUnits && j + 1 < n_tiles) ? unit_t0((j + 1) * kTUnits + lane) : -1;
        const int32_t pb_next = t0n >= 0 ? table_entry(t0n) : -1;
        const int loaded = __popc(__ballot_sync(0xffffffffu, y_cur >= 0));
        if (y_cur == -2) bad = true;
        if (j >= SK &&
            !mbar_wait_bounded(smem_u32(&k_empty[j % SK]), ((j / SK) - 1) & 1, kWaitLimit))
          bad = true;
        issue(&kmap, smem_u32(&k_full[j % SK]), k_addr(j), y_cur, loaded, false);
        if (j >= SV &&
            !mbar_wait_bounded(smem_u32(&v_empty[j % SV]), ((j / SV) - 1) & 1, kWaitLimit))
          bad = true;
        issue(&vmap, smem_u32(&v_full[j % SV]), v_addr(j), y_cur, loaded, true);
        y_next = page_y(t0n, pb_next);
      }
      // every copy started has landed (already waited for unless a wait ran out)
      if (lane == 0) {
        for (int t = max(0, n_tiles - SK); t < n_tiles; ++t)
          if (!mbar_wait_bounded(smem_u32(&k_full[t % SK]), (t / SK) & 1, kWaitLimit)) bad = true;
        for (int t = max(0, n_tiles - SV); t < n_tiles; ++t)
          if (!mbar_wait_bounded(smem_u32(&v_full[t % SV]), (t / SV) & 1, kWaitLimit)) bad = true;
      }
    } else if (warp >= kPrepWarp0) {
      // ============ V prep: fp16 in place (bf16 caches, scaled), unseen keys zeroed ============
      const int ct = tid - kPrepWarp0 * 32;
      const float2 up2 = make_float2(vr.up, vr.up);
      for (int j = 0; j < n_tiles; ++j) {
        if (!mbar_wait_bounded(smem_u32(&v_full[j % SV]), (j / SV) & 1, kWaitLimit)) bad = true;
        const int t0 = tile_t0(j);
        const uint32_t vt = v_addr(j);
        // a window tile wholly inside [k_lo, pos1] keeps every key
        const bool whole = j >= sink_tiles && t0 >= k_lo && t0 + kTKeys - 1 <= pos1;
        if (kConvert && whole) {
#pragma unroll 4
          for (int u = ct; u < Lay::kKVTile / 16; u += kPrepThreads) {  // 16-byte chunks
            uint4 x = ld_shared_v4(vt + u * 16);
            x.x = bf16x2_to_f16x2(x.x, up2);
            x.y = bf16x2_to_f16x2(x.y, up2);
            x.z = bf16x2_to_f16x2(x.z, up2);
            x.w = bf16x2_to_f16x2(x.w, up2);
            st_shared_v4(vt + u * 16, x);
          }
        } else if (kConvert) {
#pragma unroll 4
          for (int u = ct; u < Lay::kKVTile / 16; u += kPrepThreads) {
            // chunk u: unit u / (kVUnitBytes / 16), row (u / 8) % 16 of it
            const int kp = t0 + (u / (Lay::kVUnitBytes / 16)) * kUnitTokens + ((u >> 3) & 15);
            uint4 x = ld_shared_v4(vt + u * 16);
            if (kSinks ? !key_kept(j, kp) : (kp < k_lo || kp > pos1)) {
              x = make_uint4(0u, 0u, 0u, 0u);
            } else {
              x.x = bf16x2_to_f16x2(x.x, up2);
              x.y = bf16x2_to_f16x2(x.y, up2);
              x.z = bf16x2_to_f16x2(x.z, up2);
              x.w = bf16x2_to_f16x2(x.w, up2);
            }
            st_shared_v4(vt + u * 16, x);
          }
        } else if (!whole) {
          for (int r = ct; r < kTKeys; r += kPrepThreads) {
            const int kp = t0 + r;
            if (kSinks ? key_kept(j, kp) : (kp >= k_lo && kp <= pos1)) continue;
#pragma unroll
            for (int kb = 0; kb < Lay::kKBlocks; ++kb)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                st_shared_v4(vt + (r >> 4) * Lay::kVUnitBytes + kb * kUnitTokens * 128 +
                                 (r & 15) * 128 + c * 16,
                             make_uint4(0u, 0u, 0u, 0u));
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&v_ready[j % SV]));
      }
    } else {
      // ============ MMA warp: one thread waits and issues ============
      // (the role uses no warp-collective instruction; the other lanes wait
      // at the warp's join)
      if (lane == 0) {
        // A descriptor is built once per operand tile; a step inside the tile
        // adds its byte offset / 16 to the start-address field (shared
        // memory addresses stay below 256 KB, so the field cannot carry).
        auto issue_s = [&](int t, int j) {
          const uint64_t a0 = umma_sdesc_sw128(base + t * Lay::kQTileBytes, 16, 1024);
          const uint64_t b0 = umma_sdesc_sw128(k_addr(j), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // 16 columns a step: 32 bytes inside a 128-byte block, blocks a tile apart
            const uint64_t step = static_cast<uint64_t>(((kk >> 2) * kQT * 128 + (kk & 3) * 32) >> 4);
            static_assert(kQT == kTKeys, "Q and K tiles share their step offsets");
            umma_f16(tmem + Lay::s_col(t), a0 + step, b0 + step, kIdS, kk > 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&s_full[t]));
        };
        auto wait_k = [&](int j) {
          if (!mbar_wait_bounded(smem_u32(&k_full[j % SK]), (j / SK) & 1, kWaitLimit)) bad = true;
          tc_fence_after();
        };
        if (n_tiles > 0) {
          wait_k(0);
          issue_s(0, 0);
          issue_s(1, 0);
          umma_commit(smem_u32(&k_empty[0]));
        }
        // V(j) and K(j+1) are waited for by tile 0's softmax warps before
        // they announce P_0(j): acquiring p_full[0] orders them before the
        // products below, so this thread waits only for the two P tiles.
        for (int j = 0; j < n_tiles; ++j) {
          // V: keys are the K dimension (8-row groups 1 KB apart; a step of
          // 16 keys is one unit), head dims the N dimension (64-column blocks
          // 2 KB apart inside the unit)
          const uint64_t v0 = umma_sdesc_sw128(v_addr(j), kUnitTokens * 128, 1024);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!mbar_wait_bounded(smem_u32(&p_full[t]), j & 1, kWaitLimit)) bad = true;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTKeys / 16; ++kk) {
              const uint64_t vb = v0 + static_cast<uint64_t>((kk * Lay::kVUnitBytes) >> 4);
              umma_f16_ts(tmem + Lay::o_col(t), tmem + Lay::s_col(t) + kk * 8, vb, kIdO,
                          (j > 0 || kk > 0) ? 1u : 0u);
              // kExact: the lo parts of P, kTKeys / 2 columns after the hi parts
              if constexpr (kExact)
                umma_f16_ts(tmem + Lay::o_col(t), tmem + Lay::s_col(t) + kTKeys / 2 + kk * 8, vb,
                            kIdO, 1u);
            }
            if (j + 1 == n_tiles) umma_commit(smem_u32(&o_done[t]));  // O_t final
            if (t == 1) umma_commit(smem_u32(&v_empty[j % SV]));
            if (j + 1 < n_tiles) {
              // S_t(j+1) overwrites P_t(j) after the product above read it (one
              // issuing thread: the tensor pipe takes them in order)
              issue_s(t, j + 1);
              if (t == 1) umma_commit(smem_u32(&k_empty[(j + 1) % SK]));
            }
          }
        }
        // every product issued has completed
        if (n_tiles > 0) {
          umma_commit(smem_u32(&done_bar));
          if (!mbar_wait_bounded(smem_u32(&done_bar), 0, kWaitLimit)) bad = true;
        }
      }
      __syncwarp();
    }
    // the softmax warps' join and final barriers
    if (bad) s_bad = 1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    __syncthreads();
    return;
  }

  // ================= softmax warps: one row per thread =================
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
  const int t = wg;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + Lay::s_col(t) + lane_off;
  const uint32_t tO = tmem + Lay::o_col(t) + lane_off;
  // a positive scale lets the maximum be taken on the raw scores and the
  // scaling ride in the exponent's FFMA; otherwise scores are scaled first
  const bool raw_max = p.scale_log2 > 0.f;
  const float sl = raw_max ? p.scale_log2 : 1.f;
  float m_run = -INFINITY, l_run = 0.f;
  for (int j = 0; j < n_tiles; ++j) {
    const int t0 = kSinks ? tile_t0(j) : (win_u0 + j * kTUnits) * kUnitTokens;
    if (!mbar_wait_bounded(smem_u32(&s_full[t]), j & 1, kWaitLimit)) bad = true;
    tc_fence_after();
    float s[kTKeys];
    tmem_ld128(tS, s);
    if (!raw_max) {
#pragma unroll
      for (int c = 0; c < kTKeys; ++c) s[c] *= p.scale_log2;
    }
    // keys this row may not see -> -inf
    // (sink tiles always take the masked path; for the window tiles the test
    // below ignores the sinks, which can only keep keys it would mask)
    const bool edge = (kSinks && j < sink_tiles) || t0 + kTKeys - 1 > rpos ||
                      (p.window > 0 && t0 <= rpos - p.window);
    if (__any_sync(0xffffffffu, edge)) {
      if constexpr (kSinks) {
        const int kend = j < sink_tiles ? sink_end : 0x7fffffff;  // past the sink section
#pragma unroll
        for (int c = 0; c < kTKeys; ++c) {
          const int kp = t0 + c;
          const bool valid = kp <= rpos && kp < kend &&
                             (p.window <= 0 || rpos - kp < p.window || kp < num_sinks);
          s[c] = valid ? s[c] : -INFINITY;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kTKeys; ++c) {
          const int kp = t0 + c;
          const bool valid = kp <= rpos && (p.window <= 0 || rpos - kp < p.window);
          s[c] = valid ? s[c] : -INFINITY;
        }
      }
    }
    float mp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mp[i] = s[i];
#pragma unroll
    for (int c = 8; c < kTKeys; ++c) mp[c & 7] = fmaxf(mp[c & 7], s[c]);
    const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                           fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * sl;
    const float m_old = m_run;
    if (mx > m_old + kTRescale) m_run = mx;
    const bool rescale = m_run != m_old && m_old != -INFINITY;
    const float alpha = rescale ? ex2(m_old - m_run) : 1.f;
    // (nothing visible yet: p = 0; kExact: weights times 2^-down_c, which the
    // normalisation by their sum cancels)
    const float neg_m = (m_run == -INFINITY ? 0.f : -m_run) - static_cast<float>(vr.down_c);

    // S_t(j) completing means O_t += P_t(j-1) V completed too (issued before it)
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float v[16];
        tmem_ld16(tO + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= alpha;
        tmem_st16(tO + c, v);
      }
    }
    // P = 2^(s*sl - m) as fp16 over the first 64 columns of S_t (kExact: bf16
    // hi parts there, lo parts over the next 64)
    float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(neg_m, neg_m);
    if constexpr (kExact) {
#pragma unroll
      for (int h = 0; h < kTKeys / 16; ++h) {
        uint32_t w[8], wl[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 x = ffma2(make_float2(s[h * 16 + 2 * i], s[h * 16 + 2 * i + 1]), sl2, nm2);
          const float2 pr = make_float2(ex2(x.x), ex2(x.y));
          acc[i & 3] = fadd2(acc[i & 3], pr);
          split_bf16x2(pr, w[i], wl[i]);
        }
        tmem_st8u(tS + h * 8, w);
        tmem_st8u(tS + kTKeys / 2 + h * 8, wl);
      }
    } else {
#pragma unroll
      for (int h = 0; h < kTKeys / 32; ++h) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = ffma2(make_float2(s[h * 32 + 2 * i], s[h * 32 + 2 * i + 1]), sl2, nm2);
          const float2 pr = make_float2(ex2(x.x), ex2(x.y));
          acc[i & 3] = fadd2(acc[i & 3], pr);
          w[i] = Mma<__half>::pack(pr.x, pr.y);
        }
        tmem_st16u(tS + h * 16, w);
      }
    }
    const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
    l_run = l_run * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
    tmem_wait_st();
    tc_fence_before();
    if (t == 0) {
      if (!mbar_wait_bounded(smem_u32(&v_ready[j % SV]), (j / SV) & 1, kWaitLimit)) bad = true;
      if (j + 1 < n_tiles &&
          !mbar_wait_bounded(smem_u32(&k_full[(j + 1) % SK]), ((j + 1) / SK) & 1, kWaitLimit))
        bad = true;
    }
    mbar_arrive(smem_u32(&p_full[t]));
  }
  if (n_tiles > 0) {
    if (!mbar_wait_bounded(smem_u32(&o_done[t]), 0, kWaitLimit)) bad = true;
    tc_fence_after();
  }

  // ---- join, then O / l to the output rows (TMEM loads are warp-wide) ----
  if (bad) s_bad = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool nan_out = s_bad != 0;
  T* dst = static_cast<T*>(p.out) + qo_row;
  // (bf16 caches: V was scaled by vr.up)
  const float inv = nan_out ? __int_as_float(0x7fc00000) : vr.down / l_run;
#pragma unroll
  for (int c = 0; c < D; c += 16) {
    float v[16];
    if (!nan_out) {
      tmem_ld16(tO + c, v);
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

template <typename T, int D, bool kSinks, bool kExact>
cudaError_t launch_one(const CUtensorMap& kmap, const CUtensorMap& vmap, const TcParams& p,
                       int num_seqs, cudaStream_t stream) {
  using Lay = TcLayout<D>;
  auto kern = prefill_tc_kernel<T, D, kSinks, kExact>;
  const int smem = 1024 + Lay::kSmemBytes;
  // per device, once: the shared-memory opt-in, and a check that the block
  // is launched with the registers the warpgroups' split hands out (a larger
  // split would leave setmaxnreg.inc waiting)
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    cudaFuncAttributes attr{};
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * kTThreads < 2 * kQT * kSoftmaxRegs + (kTThreads - 2 * kQT) * kOtherRegs)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int64_t ctas = static_cast<int64_t>(num_seqs) * p.chunks_per_seq * p.num_kv_heads *
                       p.num_head_chunks;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(kTThreads), smem, stream, kmap,
                    vmap, p);
}

// fp16 caches: one launch.  bf16 caches: the fast launch, then the kExact
// launch, in which only the CTAs of pairs the fast one left do any work.
template <typename T, int D, bool kSinks>
cudaError_t launch_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const TcParams& p,
                     int num_seqs, cudaStream_t stream) {
  cudaError_t e = launch_one<T, D, kSinks, false>(kmap, vmap, p, num_seqs, stream);
  if constexpr (__is_same(T, __nv_bfloat16)) {
    if (e == cudaSuccess) e = launch_one<T, D, kSinks, true>(kmap, vmap, p, num_seqs, stream);
  }
  return e;
}

}  // namespace

cudaError_t launch_prefill_tc(int dtype, int head_dim, const void* q, const int32_t* cu_q,
                              int num_seqs, int num_q_heads, int max_chunk, int64_t num_blocks,
                              int num_kv_heads, int block_size, const int32_t* block_tables,
                              int max_blocks, const int32_t* context_lens, int window,
                              int num_sinks, float scale, void* out, const int32_t* order,
                              const uint2* vparts, int row_blocks, uint32_t* mode,
                              const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream) {
  TcParams p{};
  p.vparts = vparts;
  p.row_blocks = row_blocks;
  p.mode = mode;
  p.q = q;
  p.out = out;
  p.cu_q = cu_q;
  p.order = order;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.num_blocks = num_blocks;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.head_chunk_log2 = prefill_heads_log2(p.group);
  p.num_head_chunks = p.group >> p.head_chunk_log2;
  const int tok_per_cta = kRowsCta >> p.head_chunk_log2;
  p.chunks_per_seq = (max_chunk + tok_per_cta - 1) / tok_per_cta;
  p.max_blocks = max_blocks;
  p.block_size = block_size;
  p.window = window;
  p.num_sinks = window > 0 ? num_sinks : 0;
  const bool sinks = p.num_sinks > 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (dtype == 1) {
    if (head_dim == 128)
      return sinks ? launch_t<__half, 128, true>(kmap, vmap, p, num_seqs, stream)
                   : launch_t<__half, 128, false>(kmap, vmap, p, num_seqs, stream);
    return sinks ? launch_t<__half, 64, true>(kmap, vmap, p, num_seqs, stream)
                 : launch_t<__half, 64, false>(kmap, vmap, p, num_seqs, stream);
  }
  if (head_dim == 128)
    return sinks ? launch_t<__nv_bfloat16, 128, true>(kmap, vmap, p, num_seqs, stream)
                 : launch_t<__nv_bfloat16, 128, false>(kmap, vmap, p, num_seqs, stream);
  return sinks ? launch_t<__nv_bfloat16, 64, true>(kmap, vmap, p, num_seqs, stream)
               : launch_t<__nv_bfloat16, 64, false>(kmap, vmap, p, num_seqs, stream);
}

}  // namespace pkv
