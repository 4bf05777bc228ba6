// Debug-mode check of a slot index array (KDA_FLAG_CHECK_INDICES): the valid
// indices (0 <= s < num_slots) of the decode, decode-conv and recurrent steps
// must be distinct, since rows sharing a slot would race on its state. Thread
// i compares its valid index with every later one; a repeat writes
// KDA_ERR_INVALID_ARG to the status word. O(B^2) reads of a small array that
// stays in L1/L2: a debugging aid, not a production path.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kCheckThreads = 256;

__global__ void __launch_bounds__(kCheckThreads) kda_check_indices_kernel(const int32_t* idx, int B, int num_slots,
                                                                          int32_t* err) {
  __shared__ int32_t tile[kCheckThreads];
  const int i = blockIdx.x * kCheckThreads + threadIdx.x;
  const int si = i < B ? idx[i] : -1;
  const bool valid = si >= 0 && si < num_slots;
  bool repeat = false;
  // later indices, a tile at a time, starting with this block's own tile
  for (int base = blockIdx.x * kCheckThreads; base < B; base += kCheckThreads) {
    __syncthreads();
    tile[threadIdx.x] = base + threadIdx.x < B ? idx[base + threadIdx.x] : -1;
    __syncthreads();
    const int n = min(kCheckThreads, B - base);
    for (int j = 0; j < n; ++j) repeat |= valid && base + j > i && tile[j] == si;
  }
  if (repeat) set_err(err, 1 /* KDA_ERR_INVALID_ARG */);
}

}  // namespace

cudaError_t launch_check_indices(const int32_t* idx, int B, int num_slots, int32_t* err, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((B + kCheckThreads - 1) / kCheckThreads);
  kda_check_indices_kernel<<<grid, kCheckThreads, 0, s>>>(idx, B, num_slots, err);
  return cudaGetLastError();
}

}  // namespace kda
