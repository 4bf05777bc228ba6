// Output-side per-head RMSNorm ("06 · linear 路线（一）" §1 and §4 (3): GLA, GDN and
// KDA drop the linear-attention normaliser and normalise each head's output):
// for every row (one token of one head, V values) y = x / sqrt(mean(x^2) + eps) * w.
//
// Pure streaming (2 bytes in and 2 out per element): 16-byte accesses, a row
// spread over V/8 lanes (8 values each), every lane keeping kIter rows' loads
// in flight before it reduces; the mean square is summed within each row's
// lane group with xor shuffles. 8 warps per CTA. y may alias x (each element is
// read before it is written, by the same thread).
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kWarps = 8;
constexpr int kIter = 4;

template <int V>
__global__ void __launch_bounds__(32 * kWarps) kda_rmsnorm_kernel(const RmsNormCall p) {
  constexpr int LPR = V / 8;        // lanes per row
  constexpr int RPW = 32 / LPR;     // rows per warp and load step
  constexpr int ROWS_PER_WARP = RPW * kIter;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, pos = lane % LPR;
  const long long base =
      (static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * ROWS_PER_WARP + sub;
  float w[8];
  {
    const float4 w0 = *reinterpret_cast<const float4*>(p.weight + pos * 8);
    const float4 w1 = *reinterpret_cast<const float4*>(p.weight + pos * 8 + 4);
    w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w; w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
  }
  uint4 raw[kIter];
#pragma unroll
  for (int it = 0; it < kIter; ++it) {
    const long long row = base + static_cast<long long>(it) * RPW;
    raw[it] = row < p.R ? *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.x) + row * V + pos * 8)
                        : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int it = 0; it < kIter; ++it) {
    const long long row = base + static_cast<long long>(it) * RPW;
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[it]);
    float x[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __low2float(h2[i]);
      x[2 * i + 1] = __high2float(h2[i]);
      ss += x[2 * i] * x[2 * i] + x[2 * i + 1] * x[2 * i + 1];
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / static_cast<float>(V) + p.eps);
    uint4 out;
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) o2[i] = __floats2bfloat162_rn(x[2 * i] * r * w[2 * i], x[2 * i + 1] * r * w[2 * i + 1]);
    if (row < p.R) *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.y) + row * V + pos * 8) = out;
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const RmsNormCall& c, cudaStream_t s) {
  if (c.R == 0) return cudaSuccess;
  const int rows_per_cta = kWarps * kIter * (32 / (c.V / 8));
  const long long grid = (c.R + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (c.V == 128) kda_rmsnorm_kernel<128><<<static_cast<unsigned>(grid), 32 * kWarps, 0, s>>>(c);
  else if (c.V == 64) kda_rmsnorm_kernel<64><<<static_cast<unsigned>(grid), 32 * kWarps, 0, s>>>(c);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace kda
