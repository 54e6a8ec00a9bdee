// pkv_noalloc.cu -- pkv_decode_noalloc: decode with a fixed, library-resident
// split-K scratch buffer instead of a cudaMalloc'ed workspace.
//
// Who needs it: callers that cannot allocate device memory at call time --
// a serving engine that has already handed all free HBM to its own KV-block
// pool, or a latency-critical loop that must not run into the device-wide
// synchronisation cudaMalloc / cudaFree can bring.  They pass inputs and
// outputs as usual; the partial results of long-context splits go to the
// buffer below.
//
// The buffer is a file-scope __device__ array: every GPU that loads the
// library holds its PKV_NOALLOC_SCRATCH_BYTES until the process exits.  In
// host code its name is only a host-side stand-in, so the device address is
// looked up once per device with cudaGetSymbolAddress (that device current,
// on the first call there) and passed to the kernels as a plain pointer.
// Every call shares the buffer and leaves its partials in it; nothing needs
// clearing (each call writes every partial it reads), but calls that overlap
// on the GPU race on it.
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch buffer on `device` (which must be current).
int scratch_on(int device, void** addr) {
  if (device < 0 || device >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    g_scratch_addr[device] = p;
  }
  *addr = g_scratch_addr[device];
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_noalloc(const void* q, int32_t num_seqs, int32_t num_q_heads,
                                  const void* k_cache, const void* v_cache,
                                  const pkv_cache_layout* layout, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t window, float scale, void* out, void* stream) {
  int rc = pkv::decode_checks(q, num_seqs, num_q_heads, k_cache, v_cache, layout, block_tables,
                              max_blocks_per_seq, context_lens, out);
  if (rc != PKV_OK) return rc;
  // 8-bit pools need row scales, which this entry point does not take
  if (layout->dtype == PKV_FP8_E4M3 || layout->dtype == PKV_INT8) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PKV_ERR_CUDA;
  pkv::DecodeParams p{};
  int ntiles = 1;
  rc = pkv::decode_plan(num_seqs, num_q_heads, layout, max_blocks_per_seq, window, 0,
                        &p.head_chunk, &p.num_head_chunks, &ntiles, &p.units_per_split,
                        &p.num_splits);
  if (rc != PKV_OK) return rc;

  if (p.num_splits > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * p.num_splits;
    const size_t o_bytes = rows * layout->head_dim * sizeof(float);
    if (o_bytes + rows * sizeof(float2) > kScratchBytes) return PKV_ERR_SCRATCH;
    void* scratch = nullptr;
    rc = scratch_on(device, &scratch);
    if (rc != PKV_OK) return rc;
    p.part_o = static_cast<float*>(scratch);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(scratch) + o_bytes);
  }
  p.q = q;
  p.out = out;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.num_blocks = layout->num_blocks;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = layout->num_kv_heads;
  p.group = num_q_heads / layout->num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = layout->block_size;
  p.window = window;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);

  cudaError_t e;
  if (layout->dtype == PKV_FLOAT32) {
    e = pkv::launch_decode_f32(layout->head_dim, p, st);
  } else {
    CUtensorMap kmap, vmap;
    rc = pkv::pool_tensor_map(&kmap, k_cache, layout);
    if (rc != PKV_OK) return rc;
    rc = pkv::pool_tensor_map(&vmap, v_cache, layout);
    if (rc != PKV_OK) return rc;
    e = pkv::launch_decode_16bit(layout->dtype, layout->head_dim, ntiles, kmap, vmap, p, st);
  }
  if (e != cudaSuccess) return pkv::status_of(e);
  if (p.num_splits > 1) {
    e = pkv::launch_combine(layout->dtype, layout->head_dim, p, st);
    if (e != cudaSuccess) return pkv::status_of(e);
  }
  return PKV_OK;
}
