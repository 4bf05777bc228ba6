// Short-T KDA recurrent step on a state-slot pool: T tokens (T <= 64) per batch
// row applied in order to the row's slot, separate q/k/v tensors, value-head
// grouping hv -> hv / (HV / H).
//
// The operation is the general fused recurrent path that the packed decode
// specialises (sglang PR #26586 summary, 功能与动机 and 实现拆解); per token it is
// the decode step: L2 norm of q and k (eps 1e-6 in the root), q scaled,
// g = -exp(A_log) softplus(a + dt_bias) per key channel, beta = sigmoid(b),
// then decay, delta read, beta, write and output on the [V, K] state.
//
// GB300 design. Like the decode kernel, one CTA of 4 warps per (row, value
// head) streams the 64 KiB state (K = V = 128) with coalesced 16-byte
// evict-first accesses, 8 rows per warp at a time, and reduces the two dot
// products of 8 rows with one transpose reduction. The difference: a group of
// 8 rows is loaded once, all T tokens are applied to it in registers, then it
// is written back, so the state crosses HBM once per T tokens instead of once
// per token. The tokens' normalised q and k, their decay factors, beta, k.q and
// the value rows are prepared once per CTA in shared memory (warp w prepares
// tokens w, w + 4, ...), where every row group reads them.
// The per-token work grows with T: from 8 tokens per row the entry point runs
// the chunk-form kernel of kda_recurrent_tc.cu instead.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kRowGroup = 8;
constexpr int kMaxT = 64;

template <int CPL>
struct Row;
template <>
struct Row<4> {
  using T = float4;
  static __device__ __forceinline__ void get(const T& v, float (&x)[4]) { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
  static __device__ __forceinline__ T make(const float (&x)[4]) { return make_float4(x[0], x[1], x[2], x[3]); }
};
template <>
struct Row<2> {
  using T = float2;
  static __device__ __forceinline__ void get(const T& v, float (&x)[2]) { x[0] = v.x; x[1] = v.y; }
  static __device__ __forceinline__ T make(const float (&x)[2]) { return make_float2(x[0], x[1]); }
};

template <int CPL>
__device__ __forceinline__ void bf16_vec(const __nv_bfloat16* p, float (&x)[CPL]) {
#pragma unroll
  for (int i = 0; i < CPL; i += 2) {
    const __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(p + i);
    x[i] = __low2float(t);
    x[i + 1] = __high2float(t);
  }
}

// Shared memory of one CTA for T tokens: q~ (normalised, scaled), k~, alpha
// ([T][K] fp32 each), v ([T][V] fp32), beta and k~.q~ ([T] each).
__host__ __device__ constexpr size_t recurrent_smem_bytes(int T, int K, int V) {
  return sizeof(float) * (static_cast<size_t>(T) * (3 * K + V) + 2 * static_cast<size_t>(T));
}

template <int K, int V>
__global__ void __launch_bounds__(kThreads) kda_recurrent_kernel(const RecurrentCall p) {
  constexpr int CPL = K / 32;  // key channels per lane
  constexpr int ROWS_PER_WARP = V / 4;
  constexpr int GROUPS = ROWS_PER_WARP / kRowGroup;
  using Vec = typename Row<CPL>::T;
  extern __shared__ __align__(16) float rsm[];
  const int T = p.T;
  float* qs = rsm;
  float* ks = qs + T * K;
  float* as = ks + T * K;
  float* vs = as + T * K;
  float* bs = vs + T * V;
  float* kqs = bs + T;

  const int unit = blockIdx.x;  // b * HV + hv
  const int b = unit / p.HV;
  const int hv = unit - b * p.HV;
  const int h = hv / (p.HV / p.H);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int col0 = lane * CPL;

  const int slot = p.indices[b];
  if (slot < 0 || slot >= p.num_slots) {
    if (slot >= p.num_slots && threadIdx.x == 0) set_err(p.err, 1 /* KDA_ERR_INVALID_ARG */);
    for (int t = 0; t < T; ++t) {
      uint32_t* o_row = reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                    (static_cast<size_t>(b) * T + t) * p.HV * V + hv * V);
      for (int i = threadIdx.x; i < V / 2; i += kThreads) o_row[i] = 0u;
    }
    return;
  }

  float* S = p.state_pool + (static_cast<size_t>(slot) * p.HV + hv) * static_cast<size_t>(V) * K;
  const int row0 = warp * ROWS_PER_WARP;

  // The first state rows are the long pole: start them before the token prep.
  Vec cur[kRowGroup];
#pragma unroll
  for (int r = 0; r < kRowGroup; ++r)
    cur[r] = __ldcs(reinterpret_cast<const Vec*>(S + static_cast<size_t>(row0 + r) * K + col0));

  const float A = expf(p.A_log[hv]);
  float dtb[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) dtb[i] = p.dt_bias[hv * K + col0 + i];
  for (int t = warp; t < T; t += 4) {
    const size_t bt = static_cast<size_t>(b) * T + t;
    float qv[CPL], kv[CPL], av[CPL];
    bf16_vec<CPL>(reinterpret_cast<const __nv_bfloat16*>(p.q) + (bt * p.H + h) * K + col0, qv);
    bf16_vec<CPL>(reinterpret_cast<const __nv_bfloat16*>(p.k) + (bt * p.H + h) * K + col0, kv);
    bf16_vec<CPL>(reinterpret_cast<const __nv_bfloat16*>(p.a) + (bt * p.HV + hv) * K + col0, av);
    float rq = 1.f, rk = 1.f;
    if (p.l2norm) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        sq += qv[i] * qv[i];
        sk += kv[i] * kv[i];
      }
      rq = rsqrtf(warp_sum(sq) + 1e-6f);
      rk = rsqrtf(warp_sum(sk) + 1e-6f);
    }
    float kq_part = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      qv[i] *= rq * p.scale;
      kv[i] *= rk;
      kq_part += kv[i] * qv[i];
      av[i] = expf(-A * softplus_f(av[i] + dtb[i]));
    }
    const float kq = warp_sum(kq_part);
    *reinterpret_cast<Vec*>(qs + t * K + col0) = Row<CPL>::make(qv);
    *reinterpret_cast<Vec*>(ks + t * K + col0) = Row<CPL>::make(kv);
    *reinterpret_cast<Vec*>(as + t * K + col0) = Row<CPL>::make(av);
    const __nv_bfloat16* vrow = reinterpret_cast<const __nv_bfloat16*>(p.v) + (bt * p.HV + hv) * V;
    for (int i = lane; i < V; i += 32) vs[t * V + i] = __bfloat162float(vrow[i]);
    if (lane == 0) {
      bs[t] = sigmoid_f(__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.b)[bt * p.HV + hv]));
      kqs[t] = kq;
    }
  }
  __syncthreads();

  const int j = (lane >> 1) & 15;  // which of the 16 reduced values this lane ends up with
  const int rj = j & 7;
#pragma unroll 1
  for (int gi = 0; gi < GROUPS; ++gi) {
    const int rbase = row0 + gi * kRowGroup;
    Vec nxt[kRowGroup];
    if (gi + 1 < GROUPS) {
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r)
        nxt[r] = __ldcs(reinterpret_cast<const Vec*>(S + static_cast<size_t>(rbase + kRowGroup + r) * K + col0));
    }
    float sd[kRowGroup][CPL];
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) Row<CPL>::get(cur[r], sd[r]);
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      float al[CPL], kv[CPL], qv[CPL];
      Row<CPL>::get(*reinterpret_cast<const Vec*>(as + t * K + col0), al);
      Row<CPL>::get(*reinterpret_cast<const Vec*>(ks + t * K + col0), kv);
      Row<CPL>::get(*reinterpret_cast<const Vec*>(qs + t * K + col0), qv);
      float red[16];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        float pk = 0.f, py = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          sd[r][i] *= al[i];
          pk += sd[r][i] * kv[i];
          py += sd[r][i] * qv[i];
        }
        red[r] = pk;
        red[r + 8] = py;
      }
      const float tot = warp_transpose_reduce16(red, lane);
      // lanes 0..15 hold (S~ k)_r for r = j; lanes 16..31 hold (S~ q)_r for r = j - 8
      const float u = bs[t] * (vs[t * V + rbase + rj] - tot);  // meaningful on lanes 0..15
      const float other = __shfl_xor_sync(0xffffffffu, j < 8 ? u : tot, 16);
      if (j >= 8 && (lane & 1) == 0) {
        __nv_bfloat16* o_row = reinterpret_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(b) * T + t) * p.HV * V + hv * V;
        o_row[rbase + rj] = __float2bfloat16_rn(tot + other * kqs[t]);
      }
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        const float ur = __shfl_sync(0xffffffffu, u, 2 * r);
#pragma unroll
        for (int i = 0; i < CPL; ++i) sd[r][i] += ur * kv[i];
      }
    }
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r)
      __stcs(reinterpret_cast<Vec*>(S + static_cast<size_t>(rbase + r) * K + col0), Row<CPL>::make(sd[r]));
    if (gi + 1 < GROUPS) {
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) cur[r] = nxt[r];
    }
  }
}

template <int K, int V>
cudaError_t launch_recurrent_t(const RecurrentCall& c, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  {
    const cudaError_t e = set_smem_limit_once(kda_recurrent_kernel<K, V>, recurrent_smem_bytes(kMaxT, K, V), smem_set);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = static_cast<unsigned>(c.B) * static_cast<unsigned>(c.HV);
  kda_recurrent_kernel<K, V><<<grid, kThreads, recurrent_smem_bytes(c.T, K, V), s>>>(c);
  return cudaGetLastError();
}

}  // namespace

// A few tokens per row: the per-token kernel streams the state once for
// all of them and wins; from 8 tokens the chunk form on the tensor cores does.
cudaError_t launch_recurrent(const RecurrentCall& c, cudaStream_t s) {
  return c.T >= 8 ? launch_recurrent_tc(c, s) : launch_recurrent_fma(c, s);
}

cudaError_t launch_recurrent_fma(const RecurrentCall& c, cudaStream_t s) {
  if (c.B == 0) return cudaSuccess;
  if (c.T < 1 || c.T > kMaxT) return cudaErrorInvalidValue;
  if (c.K == 128 && c.V == 128) return launch_recurrent_t<128, 128>(c, s);
  if (c.K == 128 && c.V == 64) return launch_recurrent_t<128, 64>(c, s);
  if (c.K == 64 && c.V == 128) return launch_recurrent_t<64, 128>(c, s);
  if (c.K == 64 && c.V == 64) return launch_recurrent_t<64, 64>(c, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
