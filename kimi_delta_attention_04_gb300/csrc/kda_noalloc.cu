// kda_chunk_fwd_noalloc: the chunk forward on a scratch buffer the library owns,
// for callers that cannot allocate device memory when they run attention (see
// include/kda.h for who they are and the rules of use).
//
// The scratch is one file-scope __device__ array; every GPU that loads the
// library holds a copy of it until the process exits. Host code may not use
// the array's name as a device address (in host code it names a host-side
// shadow), so the first call on each device resolves the device address with
// cudaGetSymbolAddress while that device is current, and later calls reuse it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the current device's copy of the scratch, or nullptr.
void* scratch_for_current_device(kda_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *st = KDA_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = KDA_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *st = KDA_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const kda_chunk_args* args, kda_stream_t stream) {
  const size_t need = kda_chunk_workspace_size(args);
  if (need == 0) return kda_chunk_fwd(args, nullptr, 0, stream);  // reports the argument error, launches nothing
  if (need > KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_TOO_LARGE;
  kda_status st = KDA_OK;
  void* scratch = scratch_for_current_device(&st);
  if (scratch == nullptr) return st;
  return kda_chunk_fwd(args, scratch, KDA_NOALLOC_SCRATCH_BYTES, stream);
}
