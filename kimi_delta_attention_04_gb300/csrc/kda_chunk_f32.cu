// Chunkwise KDA forward, fp32 inputs, CUDA-core fp32 path (dk, dv in {64, 128}).
//
// Same algorithm and record structure as the tensor-core path (see
// kda_chunk_tc.cu): a token-parallel prep kernel builds, per (16-token chunk,
// head), q_dec, -W = -INV diag(beta) k_dec, k_res, U~ = INV diag(beta) v,
// Mqk and gamma, with L and Mqk formed from the anchored decay products of the
// level split and INV = (I + L)^{-1} from the Neumann product
// (I+X)(I+X^2)(I+X^4)(I+X^8), X = -L ("FlashKDA里的L矩阵和Mqk矩阵", sections
// L矩阵的构造, Mqk矩阵的构造, 为什么CHUNK=16); a recurrence kernel then runs
// the serial chunk loop U = U~ - W S, O = q_dec S + Mqk U,
// S = diag(gamma) S + k_res^T U (section K2 内核如何消费). Every product is an
// fp32 FMA, which is what the 1e-4 absolute tolerance of fp32 inputs needs
// (bf16/tf32 tensor-core operands cannot meet it).
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads32 = 128;
constexpr int kRecThreads32 = 256;
constexpr int kDvBlock32 = 16;

template <int DK, int DV>
struct RecF32 {
  static constexpr size_t kW = 0;                       // f32 [16][DK] (-W)
  static constexpr size_t kQd = kW + 16 * DK * 4;       // f32 [16][DK]
  static constexpr size_t kKr = kQd + 16 * DK * 4;      // f32 [16][DK]
  static constexpr size_t kUt = kKr + 16 * DK * 4;      // f32 [DV][16]
  static constexpr size_t kMqk = kUt + DV * 16 * 4;     // f32 [16][16]
  static constexpr size_t kGamma = kMqk + 16 * 16 * 4;  // f32 [DK]
  static constexpr size_t kBytes = kGamma + DK * 4;
};

template <int DK>
struct PrepSmem32 {
  float A[16][DK + 1];  // rows 0-7 k*F, rows 8-15 q*F of the row tokens of one level
  float B[8][DK + 1];   // k*F of the column tokens of one level
  float Lm[16][17];
  float Mq[16][17];
  float X[4][16][17];
  float invp[16][17];
  float red[4][48];
  float rnq[16], rnk[16], beta[16];
};

// C = (A [+ I]) (B [+ I]), 16x16, row stride 17, all threads of the block.
__device__ __forceinline__ void block_mm16(const float* A, bool addIA, const float* B, bool addIB, float* C) {
  for (int e = threadIdx.x; e < 256; e += blockDim.x) {
    const int i = e >> 4, j = e & 15;
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float a = A[i * 17 + m] + ((addIA && i == m) ? 1.f : 0.f);
      const float b = B[m * 17 + j] + ((addIB && m == j) ? 1.f : 0.f);
      acc = fmaf(a, b, acc);
    }
    C[i * 17 + j] = acc;
  }
  __syncthreads();
}

template <int DK, int DV, bool DELTA, bool L2N>
__global__ void __launch_bounds__(kPrepThreads32) kda_prep_f32_kernel(const ChunkCall p) {
  using R = RecF32<DK, DV>;
  __shared__ PrepSmem32<DK> sm;
  ChunkPos pos;
  if (!locate_chunk(p.geo, blockIdx.x, pos)) return;
  const int H = p.geo.H;
  const int h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool ownk = tid < DK, ownv = tid < DV;
  const int ck = ownk ? tid : 0, cv = ownv ? tid : 0;
  unsigned char* rec = p.records + (static_cast<size_t>(blockIdx.x) * H + h) * R::kBytes;

  for (int i = tid; i < 16 * 17; i += kPrepThreads32) {
    (&sm.Lm[0][0])[i] = 0.f;
    (&sm.Mq[0][0])[i] = 0.f;
  }
  if (tid < 16) {
    float bt = 0.f;
    if (DELTA && tid < pos.ntok) {
      const float raw = reinterpret_cast<const float*>(p.beta)[static_cast<size_t>(pos.tok0 + tid) * H + h];
      bt = (p.beta_mode == 1) ? sigmoid_f(raw) : raw;
    }
    sm.beta[tid] = bt;
  }
  const size_t kstride = static_cast<size_t>(H) * DK, vstride = static_cast<size_t>(H) * DV;
  const size_t kbase = (static_cast<size_t>(pos.tok0) * H + h) * DK + ck;
  const size_t vbase = (static_cast<size_t>(pos.tok0) * H + h) * DV + cv;
  const float* qp = reinterpret_cast<const float*>(p.q);
  const float* kp = reinterpret_cast<const float*>(p.k);
  const float* vp = reinterpret_cast<const float*>(p.v);
  float qv[16], kv[16], al[16], vv[16];
  const float Aexp = (p.gate_mode == 2) ? expf(p.A_log[h]) : 0.f;
  const float dtb = (p.gate_mode == 2 && ownk) ? p.dt_bias[h * DK + ck] : 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool vk = ownk && i < pos.ntok;
    const bool vvld = ownv && i < pos.ntok;
    qv[i] = vk ? qp[kbase + i * kstride] : 0.f;
    kv[i] = vk ? kp[kbase + i * kstride] : 0.f;
    vv[i] = vvld ? vp[vbase + i * vstride] : 0.f;
    float a = 1.f;
    if (vk) {
      if (p.gate_mode == 1) a = expf(p.g[kbase + i * kstride]);
      else if (p.gate_mode == 2) a = expf(-Aexp * softplus_f(p.a[kbase + i * kstride] + dtb));
      else if (p.gate_mode == 3) a = expf(p.g[(static_cast<size_t>(pos.tok0) + i) * H + h]);
    }
    al[i] = a;
  }
  {
    float red[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) red[i] = qv[i] * qv[i];
    const float t1 = warp_transpose_reduce16(red, lane);
#pragma unroll
    for (int i = 0; i < 16; ++i) red[i] = kv[i] * kv[i];
    const float t2 = warp_transpose_reduce16(red, lane);
#pragma unroll
    for (int i = 0; i < 16; ++i) red[i] = qv[i] * kv[i];
    const float t3 = warp_transpose_reduce16(red, lane);
    if ((lane & 1) == 0) {
      const int j = lane >> 1;
      sm.red[warp][j] = t1;
      sm.red[warp][16 + j] = t2;
      sm.red[warp][32 + j] = t3;
    }
  }
  __syncthreads();
  if (tid < 16) {
    float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepThreads32 / 32; ++w) {
      sq += sm.red[w][tid];
      sk += sm.red[w][16 + tid];
      sqk += sm.red[w][32 + tid];
    }
    const float rq = L2N ? rsqrtf(sq + 1e-6f) : 1.f;
    const float rk = L2N ? rsqrtf(sk + 1e-6f) : 1.f;
    sm.rnq[tid] = rq;
    sm.rnk[tid] = rk;
    sm.Mq[tid][tid] = p.scale * sqk * rq * rk;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    qv[i] *= sm.rnq[i];
    kv[i] *= sm.rnk[i];
  }
  float P[16], Rs[16];
  P[0] = al[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) P[i] = P[i - 1] * al[i];
  Rs[15] = 1.f;
#pragma unroll
  for (int i = 14; i >= 0; --i) Rs[i] = Rs[i + 1] * al[i + 1];
  if (ownk) {
    float* qd = reinterpret_cast<float*>(rec + R::kQd);
    float* kr = reinterpret_cast<float*>(rec + R::kKr);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      qd[i * DK + ck] = p.scale * qv[i] * P[i];
      kr[i * DK + ck] = kv[i] * Rs[i];
    }
    reinterpret_cast<float*>(rec + R::kGamma)[ck] = P[15];
  }
  if (!DELTA && ownv) {
    float* ut = reinterpret_cast<float*>(rec + R::kUt) + static_cast<size_t>(cv) * 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) ut[i] = vv[i];
  }

  // L and Mqk, one level of the anchored split at a time
#pragma unroll
  for (int lv = 0; lv < 4; ++lv) {
    const int s = 8 >> lv;
    if (ownk) {
#pragma unroll
      for (int blk = 0; blk < 8 / s; ++blk) {
        const int m = blk * 2 * s + s;
        float f = 1.f;
#pragma unroll
        for (int i = m; i < m + s; ++i) {
          if (i > m) f *= al[i];
          const int r = blk * s + (i - m);
          sm.A[r][ck] = kv[i] * f;
          sm.A[8 + r][ck] = qv[i] * f;
        }
        f = 1.f;
#pragma unroll
        for (int i = m - 1; i >= m - s; --i) {
          f *= al[i + 1];
          sm.B[blk * s + (i - (m - s))][ck] = kv[i] * f;
        }
      }
    }
    __syncthreads();
    {
      const int r = tid >> 3, cidx = tid & 7;  // 16 x 8 products, one per thread
      const int rr = r & 7;
      if (rr / s == cidx / s) {
        float acc = 0.f;
        for (int c = 0; c < DK; ++c) acc = fmaf(sm.A[r][c], sm.B[cidx][c], acc);
        const int i = (rr / s) * 2 * s + s + (rr % s);
        const int j = (cidx / s) * 2 * s + (cidx % s);
        if (r < 8) sm.Lm[i][j] = sm.beta[i] * acc;
        else sm.Mq[i][j] = p.scale * acc;
      }
    }
    __syncthreads();
  }
  {
    float* mq = reinterpret_cast<float*>(rec + R::kMqk);
    for (int e = tid; e < 256; e += kPrepThreads32) mq[e] = sm.Mq[e >> 4][e & 15];
  }
  if (!DELTA) return;

  float* X0 = &sm.X[0][0][0];
  float* X1 = &sm.X[1][0][0];
  float* X2 = &sm.X[2][0][0];
  float* X3 = &sm.X[3][0][0];
  for (int e = tid; e < 256; e += kPrepThreads32) X0[(e >> 4) * 17 + (e & 15)] = -sm.Lm[e >> 4][e & 15];
  __syncthreads();
  block_mm16(X0, false, X0, false, X1);  // X^2
  block_mm16(X1, false, X1, false, X2);  // X^4
  block_mm16(X0, true, X1, true, X3);    // (I+X)(I+X^2)
  block_mm16(X2, false, X2, false, X0);  // X^8
  block_mm16(X3, false, X2, true, X1);   // ... (I+X^4)
  block_mm16(X1, false, X0, true, X3);   // ... (I+X^8) = INV
  for (int e = tid; e < 256; e += kPrepThreads32) {
    const int i = e >> 4, j = e & 15;
    sm.invp[i][j] = X3[i * 17 + j] * sm.beta[j];
  }
  __syncthreads();
  // W (negated) and U~ from the columns each thread owns
  if (ownk) {
    float* w = reinterpret_cast<float*>(rec + R::kW);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc = fmaf(sm.invp[i][j], kv[j] * P[j], acc);
      w[i * DK + ck] = -acc;
    }
  }
  if (ownv) {
    float* ut = reinterpret_cast<float*>(rec + R::kUt) + static_cast<size_t>(cv) * 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc = fmaf(sm.invp[i][j], vv[j], acc);
      ut[i] = acc;
    }
  }
}

template <int DK>
struct RecSmem32 {
  float S[DK][kDvBlock32];
  float W[16][DK];
  float qd[16][DK];
  float kr[16][DK];
  float ut[kDvBlock32][16];
  float mqk[16][16];
  float gamma[DK];
  float U[16][kDvBlock32 + 1];
};

template <int DK, int DV, bool DELTA>
__global__ void __launch_bounds__(kRecThreads32) kda_recur_f32_kernel(const ChunkCall p) {
  using R = RecF32<DK, DV>;
  __shared__ RecSmem32<DK> sm;
  const int H = p.geo.H;
  const int n = blockIdx.x / H;
  const int h = blockIdx.x - n * H;
  const int dv0 = blockIdx.y * kDvBlock32;
  int ts, te, cb;
  if (!locate_seq(p.geo, n, ts, te, cb)) return;
  const int nch = (te - ts + kChunk - 1) / kChunk;
  const int tid = threadIdx.x;
  const float* h0 = p.h0 ? p.h0 + (static_cast<size_t>(n) * H + h) * DV * DK : nullptr;
  for (int e = tid; e < DK * kDvBlock32; e += kRecThreads32) {
    const int c = e / kDvBlock32, j = e % kDvBlock32;
    sm.S[c][j] = h0 ? h0[(dv0 + j) * DK + c] : 0.f;
  }
  const size_t rec_stride = static_cast<size_t>(H) * R::kBytes;
  const unsigned char* rec0 = p.records + (static_cast<size_t>(cb) * H + h) * R::kBytes;
  for (int c = 0; c < nch; ++c) {
    const unsigned char* rec = rec0 + static_cast<size_t>(c) * rec_stride;
    for (int e = tid; e < 16 * DK; e += kRecThreads32) {
      (&sm.W[0][0])[e] = DELTA ? reinterpret_cast<const float*>(rec + R::kW)[e] : 0.f;
      (&sm.qd[0][0])[e] = reinterpret_cast<const float*>(rec + R::kQd)[e];
      (&sm.kr[0][0])[e] = reinterpret_cast<const float*>(rec + R::kKr)[e];
    }
    for (int e = tid; e < kDvBlock32 * 16; e += kRecThreads32)
      (&sm.ut[0][0])[e] = reinterpret_cast<const float*>(rec + R::kUt)[static_cast<size_t>(dv0) * 16 + e];
    for (int e = tid; e < 256; e += kRecThreads32) (&sm.mqk[0][0])[e] = reinterpret_cast<const float*>(rec + R::kMqk)[e];
    for (int e = tid; e < DK; e += kRecThreads32) sm.gamma[e] = reinterpret_cast<const float*>(rec + R::kGamma)[e];
    __syncthreads();
    const int i = tid >> 4, j = tid & 15;  // (token, value column) of this thread
    {
      float u = sm.ut[j][i];
      if (DELTA) {
        for (int kc = 0; kc < DK; ++kc) u = fmaf(sm.W[i][kc], sm.S[kc][j], u);
      }
      sm.U[i][j] = u;
    }
    __syncthreads();
    {
      float o = 0.f;
      for (int kc = 0; kc < DK; ++kc) o = fmaf(sm.qd[i][kc], sm.S[kc][j], o);
      for (int m = 0; m <= i; ++m) o = fmaf(sm.mqk[i][m], sm.U[m][j], o);
      const int tok = ts + c * kChunk + i;
      if (tok < te) reinterpret_cast<float*>(p.o)[(static_cast<size_t>(tok) * H + h) * DV + dv0 + j] = o;
    }
    __syncthreads();
    for (int e = tid; e < DK * kDvBlock32; e += kRecThreads32) {
      const int cc = e / kDvBlock32, jj = e % kDvBlock32;
      float s = sm.gamma[cc] * sm.S[cc][jj];
#pragma unroll
      for (int m = 0; m < 16; ++m) s = fmaf(sm.kr[m][cc], sm.U[m][jj], s);
      sm.S[cc][jj] = s;
    }
    __syncthreads();
  }
  if (p.hT) {
    float* dst = p.hT + (static_cast<size_t>(n) * H + h) * DV * DK;
    for (int e = tid; e < DK * kDvBlock32; e += kRecThreads32) {
      const int j = e / DK, c = e % DK;
      dst[(dv0 + j) * DK + c] = sm.S[c][j];
    }
  }
}

template <int DK, int DV>
cudaError_t launch_f32_t(const ChunkCall& c, cudaStream_t s) {
  if (c.geo.max_chunks > 0) {
    dim3 grid(c.geo.max_chunks, c.geo.H);
    if (c.delta) {
      if (c.l2norm) kda_prep_f32_kernel<DK, DV, true, true><<<grid, kPrepThreads32, 0, s>>>(c);
      else kda_prep_f32_kernel<DK, DV, true, false><<<grid, kPrepThreads32, 0, s>>>(c);
    } else {
      if (c.l2norm) kda_prep_f32_kernel<DK, DV, false, true><<<grid, kPrepThreads32, 0, s>>>(c);
      else kda_prep_f32_kernel<DK, DV, false, false><<<grid, kPrepThreads32, 0, s>>>(c);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 grid(c.geo.N * c.geo.H, DV / kDvBlock32);
  if (c.delta) kda_recur_f32_kernel<DK, DV, true><<<grid, kRecThreads32, 0, s>>>(c);
  else kda_recur_f32_kernel<DK, DV, false><<<grid, kRecThreads32, 0, s>>>(c);
  return cudaGetLastError();
}

}  // namespace

size_t record_bytes_f32(int dk, int dv) {
  if (dk == 64 && dv == 64) return RecF32<64, 64>::kBytes;
  if (dk == 64 && dv == 128) return RecF32<64, 128>::kBytes;
  if (dk == 128 && dv == 64) return RecF32<128, 64>::kBytes;
  if (dk == 128 && dv == 128) return RecF32<128, 128>::kBytes;
  return 0;
}

cudaError_t launch_chunk_f32(const ChunkCall& c, cudaStream_t s) {
  if (c.dk == 64 && c.dv == 64) return launch_f32_t<64, 64>(c, s);
  if (c.dk == 64 && c.dv == 128) return launch_f32_t<64, 128>(c, s);
  if (c.dk == 128 && c.dv == 64) return launch_f32_t<128, 64>(c, s);
  if (c.dk == 128 && c.dv == 128) return launch_f32_t<128, 128>(c, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
