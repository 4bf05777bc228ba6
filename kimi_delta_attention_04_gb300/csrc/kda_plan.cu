// Varlen plan: from cu_seqlens (device), the first global 16-token chunk of
// every sequence (chunks restart at each sequence start), the chunk total, and
// a flag telling the chunk kernels whether cu_seqlens was valid (starts at 0,
// never decreases, ends at T). One CTA; an exclusive block scan per tile of
// 1024 sequences.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) kda_plan_kernel(const int32_t* cu, int N, int T, int32_t* off,
                                                                 int32_t* err) {
  __shared__ int warp_tot[kPlanThreads / 32];
  __shared__ int carry;
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    bad = (cu[0] != 0 || cu[N] != T) ? 1 : 0;
  }
  __syncthreads();
  for (int base = 0; base < N; base += kPlanThreads) {
    const int n = base + tid;
    int nc = 0;
    if (n < N) {
      const int len = cu[n + 1] - cu[n];
      if (len < 0) atomicOr(&bad, 1);
      nc = len > 0 ? (len + kChunk - 1) / kChunk : 0;
    }
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      warp_tot[lane] = wi - w;  // exclusive prefix of the warp totals
    }
    __syncthreads();
    const int excl = carry + warp_tot[warp] + incl - nc;
    if (n < N) off[n] = excl;
    __syncthreads();
    if (tid == kPlanThreads - 1) carry = excl + nc;
    __syncthreads();
  }
  if (tid == 0) {
    off[N] = carry;
    off[N + 1] = bad ? 0 : 1;
    if (bad) set_err(err, 1 /* KDA_ERR_INVALID_ARG */);
  }
}

}  // namespace

cudaError_t launch_plan(const ChunkCall& c, cudaStream_t s) {
  kda_plan_kernel<<<1, kPlanThreads, 0, s>>>(c.geo.cu_seqlens, c.geo.N, c.geo.T, c.geo.chunk_off, c.err);
  return cudaGetLastError();
}

}  // namespace kda
