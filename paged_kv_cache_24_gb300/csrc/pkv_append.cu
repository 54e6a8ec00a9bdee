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

// 8-bit pools: one warp per (token, kv head) row.  The row is quantised on
// its own; an all-zero row gets scale 1.  FP8: scale = absmax / 448, codes =
// E4M3(x * (448 / absmax)), round to nearest even, saturating.  INT8 (I8):
// scale = absmax / 127, codes = x * (127 / absmax) rounded to the nearest
// integer, ties to even, clamped to [-127, 127] (a NaN product gives 0).
// IEEE float32 divisions and products, so the codes are reproducible bit for
// bit.
template <typename Tin, int D, bool I8>
__global__ void append_q8_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                                  const int64_t* __restrict__ slots, int64_t num_tokens,
                                  uint8_t* __restrict__ k_codes, uint8_t* __restrict__ v_codes,
                                  float* __restrict__ k_scale, float* __restrict__ v_scale,
                                  int64_t num_blocks, int num_kv_heads, int block_size) {
  constexpr int PER = D / 32;  // elements per lane
  pdl_launch_dependents();
  pdl_wait_prior();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= num_tokens * num_kv_heads) return;
  const int64_t tok = row / num_kv_heads;
  const int h = static_cast<int>(row - tok * num_kv_heads);
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_blocks * block_size) return;
  const int64_t blk = slot / block_size;
  const int64_t dst_row = (blk * num_kv_heads + h) * block_size + (slot - blk * block_size);
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const Tin* src = (pass ? v : k) + row * D + lane * PER;
    float x[PER];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      x[i] = to_f32<Tin>(src[i]);
      amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    constexpr float kTop = I8 ? 127.f : 448.f;
    float scale = 1.f, inv = 1.f;
    if (amax > 0.f) {
      scale = __fdiv_rn(amax, kTop);
      inv = __fdiv_rn(kTop, amax);
    }
    uint32_t packed = 0;
    if constexpr (I8) {
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const float pr = __fmul_rn(x[i], inv);
        const int c = pr != pr ? 0 : min(max(__float2int_rn(pr), -127), 127);
        packed |= (static_cast<uint32_t>(c) & 0xffu) << (8 * i);
      }
    } else {
#pragma unroll
      for (int i = 0; i < PER; i += 2)
        packed |= f32x2_to_e4m3x2(__fmul_rn(x[i], inv), __fmul_rn(x[i + 1], inv)) << (8 * i);
    }
    uint8_t* dst = (pass ? v_codes : k_codes) + dst_row * D + lane * PER;
    if constexpr (PER == 4) {
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    }
    if (lane == 0) (pass ? v_scale : k_scale)[dst_row] = scale;
  }
}

}  // namespace

cudaError_t launch_append_q8(bool int8, int in_dtype, const void* k, const void* v,
                             const int64_t* slots, int64_t num_tokens, void* k_codes,
                             void* v_codes, float* k_scale, float* v_scale, int64_t num_blocks,
                             int num_kv_heads, int block_size, int head_dim,
                             cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int64_t rows = num_tokens * num_kv_heads;
  const int warps = 8;
  const int64_t blocks = (rows + warps - 1) / warps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto* kc = static_cast<uint8_t*>(k_codes);
  auto* vc = static_cast<uint8_t*>(v_codes);
#define PKV_APPEND8_K(T, D, I8)                                                        \
  launch_pdl(append_q8_kernel<T, D, I8>, dim3(static_cast<unsigned>(blocks)),             \
             dim3(warps * 32), 0, stream, static_cast<const T*>(k), static_cast<const T*>(v), \
             slots, num_tokens, kc, vc, k_scale, v_scale, num_blocks, num_kv_heads,       \
             block_size)
#define PKV_APPEND8(T, D) return int8 ? PKV_APPEND8_K(T, D, true) : PKV_APPEND8_K(T, D, false)
  if (in_dtype == 0) {
    if (head_dim == 128) PKV_APPEND8(float, 128);
    PKV_APPEND8(float, 64);
  }
  if (in_dtype == 1) {
    if (head_dim == 128) PKV_APPEND8(__half, 128);
    PKV_APPEND8(__half, 64);
  }
  if (head_dim == 128) PKV_APPEND8(__nv_bfloat16, 128);
  PKV_APPEND8(__nv_bfloat16, 64);
#undef PKV_APPEND8
#undef PKV_APPEND8_K
}

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
