// pkv_stage.cu -- copies of a step's staged inputs (host -> device) and of its
// output (device -> host) as a kernel: on a host whose pinned memory the GPU
// reaches by load and store over a coherent link, many threads moving 16
// bytes each finish a transfer of a few MB well before a copy-engine
// transfer of the same bytes, whose fixed cost dominates at this size.
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_stage.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
stage_copy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src, int64_t bytes) {
  pdl_launch_dependents();
  pdl_wait_prior();  // the source may be written by the previous launch
  const int64_t n16 = bytes >> 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint4* d = reinterpret_cast<uint4*>(dst);
  const uint4* s = reinterpret_cast<const uint4*>(src);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride)
    d[i] = s[i];
  if (blockIdx.x == 0 && threadIdx.x < (bytes & 15))  // the last bytes, one per thread
    dst[(n16 << 4) + threadIdx.x] = src[(n16 << 4) + threadIdx.x];
}

}  // namespace

cudaError_t launch_stage_copy(void* dst, const void* src, int64_t bytes, int num_sms,
                              cudaStream_t stream) {
  if (bytes <= 0) return cudaSuccess;
  const int64_t n16 = (bytes + 15) >> 4;
  int64_t blocks = (n16 + kCopyThreads - 1) / kCopyThreads;
  const int64_t cap = 4 * static_cast<int64_t>(num_sms > 0 ? num_sms : 148);
  if (blocks > cap) blocks = cap;
  return launch_pdl(stage_copy_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCopyThreads),
                    0, stream, static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src),
                    bytes);
}

}  // namespace pkv
