// Self-test of the bounded device-side wait that every mbarrier wait of the
// fused chunk kernel uses: one thread waits on a fresh mbarrier that nothing
// arrives on, with a short limit, and must give up, report KDA_ERR_TIMEOUT in
// the status word and return, leaving the context usable. This lets a test
// exercise the failure path without a fault or a hang.
#include "kda_cluster.cuh"
#include "kda_common.cuh"

namespace kda {
namespace {

__global__ void kda_wait_selftest_kernel(int32_t* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(smem_u32(&bar), 0u, limit_ns)) set_err(err, 4 /* KDA_ERR_TIMEOUT */);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t s) {
  kda_wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace kda
