// Fused T=1 KDA decode on a packed q|k|v row with a state-slot pool.
//
// Behaviour follows the packed decode kernel of sglang PR #26586
// (fused_recurrent_kda_packed_decode): slot lookup with -1 as padding, q/k/v
// read at their offsets in the packed row, in-kernel L2 norm (eps 1e-6 in the
// root), q scaled, g = -exp(A_log) softplus(a + dt_bias) per key channel,
// beta = sigmoid(b), then decay, delta read, beta, write and output on the
// [V, K] state of the slot, written back in place.
//
// GB300 design: the work is pure HBM streaming (64 KiB of fp32 state read and
// written per (row, value head)), so the kernel is built around keeping many
// 16-byte loads in flight, not around arithmetic:
//   * one CTA of 4 warps per (row, value head); each warp owns V/4 state rows;
//   * a lane owns K/32 consecutive key channels, so a state row is one fully
//     coalesced 512 B (K = 128) warp access; rows are read with streaming
//     (evict-first) loads, register double-buffered 8 rows at a time;
//   * the two dot products of each row (S~ k and S~ q) are reduced for 8 rows
//     at once with a transpose reduction (16 shuffles for 16 sums); the output
//     uses o_r = S~_r q + u_r (k q), so no second pass over the updated row.
// With the causal conv1d + SiLU in front (CONV), the CTA first asks L2 for its
// slot, its 128 threads convolve the row's q/k channels once between them
// (shared through shared memory) and each thread its own v channel; then the
// state stream runs as above.
#include "kda_cluster.cuh"
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kRowGroup = 8;

template <int CPL>
struct RowVec;
template <>
struct RowVec<4> {
  using T = float4;
  static __device__ __forceinline__ void get(const T& v, float (&x)[4]) { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
  static __device__ __forceinline__ T make(const float (&x)[4]) { return make_float4(x[0], x[1], x[2], x[3]); }
};
template <>
struct RowVec<2> {
  using T = float2;
  static __device__ __forceinline__ void get(const T& v, float (&x)[2]) { x[0] = v.x; x[1] = v.y; }
  static __device__ __forceinline__ T make(const float (&x)[2]) { return make_float2(x[0], x[1]); }
};

template <int CPL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float (&x)[CPL]) {
#pragma unroll
  for (int i = 0; i < CPL; i += 2) {
    __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(p + i);
    x[i] = __low2float(t);
    x[i + 1] = __high2float(t);
  }
}

// Causal conv1d + SiLU of one channel c of a row ("关键源码片段",
// KDAAttnBackend.forward_decode: causal_conv1d_update before the packed decode):
// window = [conv state (W-1 inputs, oldest first); x], y = silu(w . window + b).
// When `write`, the slot's state becomes window[1:] (exact bf16 copies).
__device__ __forceinline__ float conv_silu(const DecodeCall& p, int slot, int b, int C, int c, bool write) {
  const int W = p.conv_W;
  const __nv_bfloat16* in = reinterpret_cast<const __nv_bfloat16*>(p.conv_in) + static_cast<size_t>(slot) * (W - 1) * C;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.conv_out) + static_cast<size_t>(slot) * (W - 1) * C;
  const __nv_bfloat16 x = reinterpret_cast<const __nv_bfloat16*>(p.packed_qkv)[static_cast<size_t>(b) * C + c];
  float acc = p.conv_b ? p.conv_b[c] : 0.f;
  __nv_bfloat16 win[3];
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (i < W - 1) {
      win[i] = in[static_cast<size_t>(i) * C + c];
      acc += p.conv_w[static_cast<size_t>(c) * W + i] * __bfloat162float(win[i]);
    }
  acc += p.conv_w[static_cast<size_t>(c) * W + W - 1] * __bfloat162float(x);
  if (write) {
#pragma unroll
    for (int i = 0; i < 3; ++i)
      if (i < W - 1) out[static_cast<size_t>(i) * C + c] = (i + 1 < W - 1) ? win[i + 1] : x;
  }
  return acc / (1.f + expf(-acc));
}

// The state shift of conv_silu alone (window[1:] into the slot), for channels
// whose output was computed by several threads that all had to read first.
__device__ __forceinline__ void conv_shift(const DecodeCall& p, int slot, int b, int C, int c) {
  const int W = p.conv_W;
  const __nv_bfloat16* in = reinterpret_cast<const __nv_bfloat16*>(p.conv_in) + static_cast<size_t>(slot) * (W - 1) * C;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.conv_out) + static_cast<size_t>(slot) * (W - 1) * C;
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (i < W - 1)
      out[static_cast<size_t>(i) * C + c] =
          (i + 1 < W - 1) ? in[static_cast<size_t>(i + 1) * C + c]
                          : reinterpret_cast<const __nv_bfloat16*>(p.packed_qkv)[static_cast<size_t>(b) * C + c];
}

template <int K, int V, bool CONV>
__global__ void __launch_bounds__(kDecodeThreads) kda_decode_kernel(const DecodeCall p) {
  constexpr int CPL = K / 32;                 // key channels per lane
  constexpr int ROWS_PER_WARP = V / 4;
  constexpr int GROUPS = ROWS_PER_WARP / kRowGroup;
  using Vec = typename RowVec<CPL>::T;

  const int unit = blockIdx.x;  // b * HV + hv
  const int b = unit / p.HV;
  const int hv = unit - b * p.HV;
  const int h = hv / (p.HV / p.H);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  __nv_bfloat16* o_row = reinterpret_cast<__nv_bfloat16*>(p.o) + static_cast<size_t>(unit) * V;
  const int slot = p.indices[b];
  if (slot < 0 || slot >= p.num_slots) {
    if (slot >= p.num_slots && threadIdx.x == 0) set_err(p.err, 1 /* KDA_ERR_INVALID_ARG */);
    for (int i = threadIdx.x; i < V / 2; i += kDecodeThreads) reinterpret_cast<uint32_t*>(o_row)[i] = 0u;
    return;
  }

  float* S = p.state_pool + (static_cast<size_t>(slot) * p.HV + hv) * static_cast<size_t>(V) * K;
  const int row0 = warp * ROWS_PER_WARP;
  const int col0 = lane * CPL;

  // With the conv in front, the stream below waits for the conv's loads and a
  // barrier: the whole slot is asked of L2 first, so the stream then hits L2.
  if (CONV && threadIdx.x == 0) {
    constexpr uint32_t kPart = 16384;
    for (uint32_t off = 0; off < static_cast<uint32_t>(V * K * 4); off += kPart)
      bulk_prefetch_l2(reinterpret_cast<const unsigned char*>(S) + off, kPart);
  }
  // Start the first state rows before anything else: they are the long pole.
  Vec cur[kRowGroup];
#pragma unroll
  for (int r = 0; r < kRowGroup; ++r)
    cur[r] = __ldcs(reinterpret_cast<const Vec*>(S + static_cast<size_t>(row0 + r) * K + col0));

  const int C = 2 * p.H * K + p.HV * V;
  const __nv_bfloat16* row = reinterpret_cast<const __nv_bfloat16*>(p.packed_qkv) + static_cast<size_t>(b) * C;
  float qv[CPL], kv[CPL], av[CPL];
  __shared__ float vconv[CONV ? V : 1];
  __shared__ __align__(16) float qkconv[CONV ? 2 * K : 4];
  if (CONV) {
    // Every warp needs the whole q and k (they differ only in state rows): the
    // CTA's threads convolve the 2K q/k channels once between them and share
    // them through shared memory. A q/k channel is also read by the other value
    // heads of its group, so all convolve from the old state first; after the
    // barrier, warp 0 of the group's first value head writes the new q/k state.
    // Each v channel has one owning thread, which reads and writes it.
    for (int c = threadIdx.x; c < 2 * K; c += kDecodeThreads)
      qkconv[c] = conv_silu(p, slot, b, C, (c < K ? h * K + c : p.H * K + h * K + c - K), false);
    for (int r = threadIdx.x; r < V; r += kDecodeThreads) vconv[r] = conv_silu(p, slot, b, C, 2 * p.H * K + hv * V + r, true);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      qv[i] = qkconv[col0 + i];
      kv[i] = qkconv[K + col0 + i];
    }
    if (warp == 0 && hv % (p.HV / p.H) == 0) {
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        conv_shift(p, slot, b, C, h * K + col0 + i);
        conv_shift(p, slot, b, C, p.H * K + h * K + col0 + i);
      }
    }
  } else {
    load_bf16<CPL>(row + h * K + col0, qv);
    load_bf16<CPL>(row + p.H * K + h * K + col0, kv);
  }
  load_bf16<CPL>(reinterpret_cast<const __nv_bfloat16*>(p.a) + static_cast<size_t>(b) * p.HV * K + hv * K + col0, av);
  const __nv_bfloat16* vrow = row + 2 * p.H * K + hv * V;

  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    sq += qv[i] * qv[i];
    sk += kv[i] * kv[i];
  }
  float rq = 1.f, rk = 1.f;
  if (p.l2norm) {
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    rq = rsqrtf(sq + 1e-6f);
    rk = rsqrtf(sk + 1e-6f);
  }
  const float A = expf(p.A_log[hv]);
  const float beta = sigmoid_f(__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.b)[static_cast<size_t>(b) * p.HV + hv]));
  float alpha[CPL], kq_part = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    qv[i] *= rq * p.scale;
    kv[i] *= rk;
    kq_part += kv[i] * qv[i];
    alpha[i] = expf(-A * softplus_f(av[i] + p.dt_bias[hv * K + col0 + i]));
  }
  const float kq = warp_sum(kq_part);
  const int j = (lane >> 1) & 15;  // which of the 16 reduced values this lane ends up with
  const int rj = j & 7;

#pragma unroll
  for (int gi = 0; gi < GROUPS; ++gi) {
    const int rbase = row0 + gi * kRowGroup;
    Vec nxt[kRowGroup];
    if (gi + 1 < GROUPS) {
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r)
        nxt[r] = __ldcs(reinterpret_cast<const Vec*>(S + static_cast<size_t>(rbase + kRowGroup + r) * K + col0));
    }
    const float vr = CONV ? vconv[rbase + rj] : __bfloat162float(vrow[rbase + rj]);

    float sd[kRowGroup][CPL];
    float red[16];
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) {
      RowVec<CPL>::get(cur[r], sd[r]);
      float pk = 0.f, py = 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        sd[r][i] *= alpha[i];
        pk += sd[r][i] * kv[i];
        py += sd[r][i] * qv[i];
      }
      red[r] = pk;
      red[r + 8] = py;
    }
    const float tot = warp_transpose_reduce16(red, lane);
    // lanes 0..15 hold (S~ k)_r for r = j; lanes 16..31 hold (S~ q)_r for r = j - 8
    const float u = beta * (vr - tot);  // meaningful on lanes 0..15
    const float other = __shfl_xor_sync(0xffffffffu, j < 8 ? u : tot, 16);
    if (j >= 8 && (lane & 1) == 0) {
      const float o_r = tot + other * kq;
      o_row[rbase + rj] = __float2bfloat16_rn(o_r);
    }
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) {
      const float ur = __shfl_sync(0xffffffffu, u, 2 * r);
      float nw[CPL];
#pragma unroll
      for (int i = 0; i < CPL; ++i) nw[i] = sd[r][i] + ur * kv[i];
      __stcs(reinterpret_cast<Vec*>(S + static_cast<size_t>(rbase + r) * K + col0), RowVec<CPL>::make(nw));
    }
    if (gi + 1 < GROUPS) {
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) cur[r] = nxt[r];
    }
  }
}

template <int K, int V>
cudaError_t launch_decode_t(const DecodeCall& c, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(c.B) * static_cast<unsigned>(c.HV);
  if (c.conv_in != nullptr) kda_decode_kernel<K, V, true><<<grid, kDecodeThreads, 0, s>>>(c);
  else kda_decode_kernel<K, V, false><<<grid, kDecodeThreads, 0, s>>>(c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeCall& c, cudaStream_t s) {
  if (c.B == 0) return cudaSuccess;
  if (c.K == 128 && c.V == 128) return launch_decode_t<128, 128>(c, s);
  if (c.K == 128 && c.V == 64) return launch_decode_t<128, 64>(c, s);
  if (c.K == 64 && c.V == 128) return launch_decode_t<64, 128>(c, s);
  if (c.K == 64 && c.V == 64) return launch_decode_t<64, 64>(c, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
