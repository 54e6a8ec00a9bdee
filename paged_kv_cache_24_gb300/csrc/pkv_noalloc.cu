// pkv_noalloc.cu -- the fixed split-K scratch buffer of pkv_decode_noalloc and
// pkv_decode_noalloc_ex (the entry points themselves are in pkv_api.cu).
//
// Who needs it: callers that cannot allocate device memory at call time --
// a serving engine that has already handed all free HBM to its own KV-block
// pool, or a latency-critical loop that must not run into the device-wide
// synchronisation cudaMalloc / cudaFree can bring.  The partial results of
// long-context splits go to the buffer below instead of a cudaMalloc'ed
// workspace.
//
// The buffer is a file-scope __device__ array: every GPU that loads the
// library holds its PKV_NOALLOC_SCRATCH_BYTES until the process exits.  In
// host code its name is only a host-side stand-in, so the device address is
// looked up once per device with cudaGetSymbolAddress (that device current,
// on the first call there) and passed to the kernels as a plain pointer.
// pkv_release_workspaces forgets the looked-up addresses, so that after a
// device reset (which reloads the library's device image) the next call looks
// the buffer up again instead of using a stale address.
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

}  // namespace

namespace pkv {

int noalloc_scratch(int device, void** addr) {
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

void noalloc_forget() {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  for (void*& a : g_scratch_addr) a = nullptr;
}

}  // namespace pkv
