// Chunkwise KDA forward, bf16 inputs, tensor-core path (mma.sync m16n8k16,
// fp32 accumulation) for dk = dv = D in {64, 128}.
//
// Two kernels per call:
//
// 1. prep (token-parallel, one CTA per (16-token chunk, head)) computes, from
//    "FlashKDA里的L矩阵和Mqk矩阵" (sections L矩阵的构造, Mqk矩阵的构造,
//    为什么CHUNK=16, K2 内核如何消费):
//      q, k L2-normalised (optional), alpha = e^g (g given, zero, or
//      -exp(A_log) softplus(a + dt_bias)), beta (given or sigmoid of logits);
//      P_i = prod_{t<=i} alpha_t   (= e^{G_i}, G the in-chunk inclusive cumsum)
//      q_dec = scale q P,  k_dec = k P,  k_res_j = k_j prod_{t>j} alpha_t,  gamma = P_15
//      L[i,j]   = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}   (j < i)
//      Mqk[i,j] = scale  sum_c q_ic k_jc e^{G_ic - G_jc}   (j <= i)
//      INV = (I + L)^{-1} by the Neumann product (I+X)(I+X^2)(I+X^4)(I+X^8), X = -L
//      W = INV diag(beta) k_dec,  U~ = INV diag(beta) v          (WY form)
//    and stores one record per (chunk, head) in the workspace.
//    The pair factors e^{G_i - G_j} are never formed as e^{G_i} e^{-G_j} (that
//    overflows fp32 once -G > 88, which these gates reach inside one chunk).
//    Instead each strictly-lower pair (i, j) belongs to exactly one level of a
//    binary split of the chunk (block sizes 8, 4, 2, 1): at that level i lies
//    in the upper and j in the lower half of one block with anchor m = the
//    first row of the upper half, and e^{G_i - G_j} = [prod_{m<t<=i} alpha_t]
//    [prod_{j<t<=m} alpha_t]: two factors <= 1, products of alpha only. Per
//    level the 8 "row" tokens (upper halves) and 8 "column" tokens (lower
//    halves) give one 16x8x(dk) MMA that yields the L and Mqk entries of that
//    level at once (rows 0-7: k rows, rows 8-15: q rows).
//
// 2. recurrence (one CTA per (sequence, head, 16*WARPS value rows); each warp
//    owns 16 value rows of the state, S^T [16 x dk] fp32 in registers as the
//    m16n8 accumulators) runs the serial chunk loop:
//      U^T  = U~^T - S^T W^T          (S^T as the bf16 A operand)
//      O^T  = S^T q_dec^T + U^T Mqk^T (U^T as the A operand, no shuffles)
//      S^T  = S^T diag(gamma) + U^T k_res
//    i.e. "out = q_dec S + Mqk U; S = e^{g_total} S + k_res^T U" of the K2
//    section, with the inverse folded into W / U~ so that only two dependent
//    MMA stages sit on the serial path. Chunk operands are staged in shared
//    memory by cp.async, double buffered.
//
// Operand precision: S, W, q_dec bf16; U, k_res, Mqk fp16 with the delta rule
// on (bf16 when off, where U = v is exact in bf16); L/Mqk/INV operands fp16
// when q and k are L2-normalised (all entries bounded by 1), bf16 otherwise;
// U~ is kept in fp32.
#include <type_traits>

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads = 128;

template <int D>
struct RecTC {
  static constexpr size_t kW = 0;                        // bf16 [16][D]  (-W)
  static constexpr size_t kQd = kW + 16 * D * 2;         // bf16 [16][D]
  static constexpr size_t kKr = kQd + 16 * D * 2;        // st2  [16][D]
  static constexpr size_t kUt = kKr + 16 * D * 2;        // f32  [D][16]  (U~ transposed)
  static constexpr size_t kMqk = kUt + D * 16 * 4;       // st2  [16][16]
  static constexpr size_t kGamma = kMqk + 16 * 16 * 2;   // f32  [D]
  static constexpr size_t kBytes = kGamma + D * 4;
  static_assert(kBytes % 16 == 0, "record must keep 16-byte alignment");
};

template <int D, typename Q>
struct PrepSmem {
  __align__(16) Q A_lv[4][16][D + 8];   // per level: rows 0-7 k*F, rows 8-15 q*F of the row tokens
  __align__(16) Q B_lv[4][8][D + 8];    // per level: k*F of the column tokens
  __align__(16) Q kdec[16][D + 8];
  __align__(16) __nv_bfloat16 vs[16][D + 8];
  __align__(16) Q invq[16][24];
  __align__(16) __nv_bfloat16 invhi[16][24];
  __align__(16) __nv_bfloat16 invlo[16][24];
  float Lm[16][17];
  float Mq[16][17];
  float X[4][16][17];
  float red[4][48];
  float rnq[16], rnk[16], beta[16];
};

// Row / column token of slot r at a level with half-block size s.
// Token of row r (column r) of a level's 8-row block, the level's half-block size
// being s = 2^ls (shifts: the level is a warp index, so a division would be a
// run-time one).
__device__ __forceinline__ int row_tok(int ls, int r) { return ((r >> ls) << (ls + 1)) + (1 << ls) + (r & ((1 << ls) - 1)); }
__device__ __forceinline__ int col_tok(int ls, int r) { return ((r >> ls) << (ls + 1)) + (r & ((1 << ls) - 1)); }

// C = (A [+ I]) (B [+ I]) for 16x16 fp32 matrices in shared memory (row stride
// 17), one warp, operands rounded to Op; C must not alias A or B.
template <typename Op>
__device__ __forceinline__ void warp_mm16(const float* A, bool addIA, const float* B, bool addIB, float* C,
                                          int lane) {
  const int g = lane >> 2, t = lane & 3;
  auto ea = [&](int r, int c) { return A[r * 17 + c] + ((addIA && r == c) ? 1.f : 0.f); };
  auto eb = [&](int r, int c) { return B[r * 17 + c] + ((addIB && r == c) ? 1.f : 0.f); };
  uint32_t a[4];
  a[0] = Op::pack(ea(g, 2 * t), ea(g, 2 * t + 1));
  a[1] = Op::pack(ea(g + 8, 2 * t), ea(g + 8, 2 * t + 1));
  a[2] = Op::pack(ea(g, 2 * t + 8), ea(g, 2 * t + 9));
  a[3] = Op::pack(ea(g + 8, 2 * t + 8), ea(g + 8, 2 * t + 9));
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int n = 8 * nt + g;
    const uint32_t b0 = Op::pack(eb(2 * t, n), eb(2 * t + 1, n));
    const uint32_t b1 = Op::pack(eb(2 * t + 8, n), eb(2 * t + 9, n));
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816<Op>(c, a, b0, b1);
    const int col = 8 * nt + 2 * t;
    C[g * 17 + col] = c[0];
    C[g * 17 + col + 1] = c[1];
    C[(g + 8) * 17 + col] = c[2];
    C[(g + 8) * 17 + col + 1] = c[3];
  }
  __syncwarp();
}

template <int D, bool DELTA, bool L2N>
__global__ void __launch_bounds__(kPrepThreads) kda_prep_tc_kernel(const ChunkCall p) {
  using QK = std::conditional_t<L2N, F16, Bf16>;
  using ST2 = std::conditional_t<DELTA, F16, Bf16>;
  using Q = typename QK::T;
  using R = RecTC<D>;
  __shared__ PrepSmem<D, Q> sm;

  ChunkPos pos;
  if (!locate_chunk(p.geo, blockIdx.x, pos)) return;
  const int H = p.geo.H;
  const int h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool own = tid < D;
  const int ch = own ? tid : 0;
  unsigned char* rec = p.records + (static_cast<size_t>(blockIdx.x) * H + h) * R::kBytes;

  for (int i = tid; i < 16 * 17; i += kPrepThreads) {
    (&sm.Lm[0][0])[i] = 0.f;
    (&sm.Mq[0][0])[i] = 0.f;
  }
  if (tid < 16) {
    float bt = 0.f;
    if (DELTA && tid < pos.ntok) {
      const float raw = __bfloat162float(
          reinterpret_cast<const __nv_bfloat16*>(p.beta)[static_cast<size_t>(pos.tok0 + tid) * H + h]);
      bt = (p.beta_mode == 1) ? sigmoid_f(raw) : raw;
    }
    sm.beta[tid] = bt;
  }

  // ---- the chunk's rows of q, k, v and the per-channel gate, staged in shared
  // memory with 16-byte cp.async (the level-operand buffers are free until the
  // operands are written, two barriers later); rows past the chunk are zeroed ----
  struct StagedIn {
    __nv_bfloat16 q[16][D];
    __nv_bfloat16 k[16][D];
    __nv_bfloat16 v[16][D];
    float g[16][D];  // g (gate mode 1) or the gate input a (mode 2)
  };
  static_assert(sizeof(StagedIn) <= sizeof(sm.A_lv) + sizeof(sm.B_lv), "staging fits the level buffers");
  StagedIn& in = *reinterpret_cast<StagedIn*>(&sm.A_lv[0][0][0]);
  const bool gate_rows = p.gate_mode == 1 || p.gate_mode == 2;
  {
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(p.v);
    const float* gb = p.gate_mode == 1 ? p.g : p.a;
    constexpr int V8 = D / 8, V4 = D / 4;  // 16-byte vectors per bf16 / fp32 row
    for (int i = tid; i < 16 * V8; i += kPrepThreads) {
      const int row = i / V8, c8 = i - row * V8;
      if (row < pos.ntok) {
        const size_t off = (static_cast<size_t>(pos.tok0 + row) * H + h) * D + c8 * 8;
        cp_async16(&in.q[row][c8 * 8], qb + off);
        cp_async16(&in.k[row][c8 * 8], kb + off);
        cp_async16(&in.v[row][c8 * 8], vb + off);
      } else {
        *reinterpret_cast<uint4*>(&in.q[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(&in.k[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(&in.v[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
      }
    }
    if (gate_rows) {
      for (int i = tid; i < 16 * V4; i += kPrepThreads) {
        const int row = i / V4, c4 = i - row * V4;
        if (row < pos.ntok) cp_async16(&in.g[row][c4 * 4], gb + (static_cast<size_t>(pos.tok0 + row) * H + h) * D + c4 * 4);
        else *reinterpret_cast<float4*>(&in.g[row][c4 * 4]) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
  }
  __syncthreads();

  // ---- per-channel columns of the chunk (thread ch owns key channel ch) ----
  float qv[16], kv[16], al[16], vv[16];
  const float Aexp = (p.gate_mode == 2) ? expf(p.A_log[h]) : 0.f;
  const float dtb = (p.gate_mode == 2 && own) ? p.dt_bias[h * D + ch] : 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool valid = own && i < pos.ntok;
    qv[i] = valid ? __bfloat162float(in.q[i][ch]) : 0.f;
    kv[i] = valid ? __bfloat162float(in.k[i][ch]) : 0.f;
    vv[i] = valid ? __bfloat162float(in.v[i][ch]) : 0.f;
    float a = 1.f;
    if (valid) {
      if (p.gate_mode == 1) {
        a = expf(in.g[i][ch]);
      } else if (p.gate_mode == 2) {
        const float x = in.g[i][ch] + dtb;
        a = expf(-Aexp * softplus_f(x));
      } else if (p.gate_mode == 3) {  // one decay per token and head
        a = expf(p.g[(static_cast<size_t>(pos.tok0) + i) * H + h]);
      }
    }
    al[i] = a;
  }

  // ---- row sums of q^2, k^2 and q.k over the channels ----
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
    for (int w = 0; w < kPrepThreads / 32; ++w) {
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

  // ---- decay products, record operands, level operands ----
  float P[16], Rs[16];
  P[0] = al[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) P[i] = P[i - 1] * al[i];
  Rs[15] = 1.f;
#pragma unroll
  for (int i = 14; i >= 0; --i) Rs[i] = Rs[i + 1] * al[i + 1];

  if (own) {
    __nv_bfloat16* qd = reinterpret_cast<__nv_bfloat16*>(rec + R::kQd);
    typename ST2::T* kr = reinterpret_cast<typename ST2::T*>(rec + R::kKr);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      qd[i * D + ch] = __float2bfloat16_rn(p.scale * qv[i] * P[i]);
      kr[i * D + ch] = ST2::cvt(kv[i] * Rs[i]);
      if (DELTA) {
        sm.kdec[i][ch] = QK::cvt(kv[i] * P[i]);
        sm.vs[i][ch] = __float2bfloat16_rn(vv[i]);
      }
    }
    reinterpret_cast<float*>(rec + R::kGamma)[ch] = P[15];
    if (!DELTA) {  // U = v exactly
      float4* ut = reinterpret_cast<float4*>(rec + R::kUt + static_cast<size_t>(ch) * 16 * 4);
#pragma unroll
      for (int i = 0; i < 16; i += 4) ut[i / 4] = make_float4(vv[i], vv[i + 1], vv[i + 2], vv[i + 3]);
    }
#pragma unroll
    for (int lv = 0; lv < 4; ++lv) {
      const int s = 8 >> lv;
#pragma unroll
      for (int blk = 0; blk < 8 / s; ++blk) {
        const int m = blk * 2 * s + s;  // anchor: first row of the upper half
        float f = 1.f;
#pragma unroll
        for (int i = m; i < m + s; ++i) {  // row tokens: prod_{m<t<=i} alpha_t
          if (i > m) f *= al[i];
          const int r = blk * s + (i - m);
          if (DELTA) sm.A_lv[lv][r][ch] = QK::cvt(kv[i] * f);
          sm.A_lv[lv][8 + r][ch] = QK::cvt(qv[i] * f);
        }
        f = 1.f;
#pragma unroll
        for (int i = m - 1; i >= m - s; --i) {  // column tokens: prod_{i<t<=m} alpha_t
          f *= al[i + 1];
          const int r = blk * s + (i - (m - s));
          sm.B_lv[lv][r][ch] = QK::cvt(kv[i] * f);
        }
      }
    }
  }
  __syncthreads();

  // ---- L and Mqk: warp lv multiplies the operands of level lv ----
  {
    const int lv = warp;
    const int ls = 3 - lv;  // half-block size 2^ls = 8 >> lv
    // Without the delta rule rows 0-7 (k rows) are never written and their
    // results are discarded; MMA rows are independent, so they cannot leak.
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4], b[2];
      ldsm_x4(a, &sm.A_lv[lv][lane & 15][16 * kk + (lane >> 4) * 8]);
      ldsm_x2(b, &sm.B_lv[lv][lane & 7][16 * kk + ((lane >> 3) & 1) * 8]);
      mma16816<QK>(acc, a, b[0], b[1]);
    }
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = g + ((e & 2) ? 8 : 0);
      const int cidx = 2 * t + (e & 1);
      const int rr = r & 7;
      if ((rr >> ls) != (cidx >> ls)) continue;  // not a pair of this level
      const int i = row_tok(ls, rr), j = col_tok(ls, cidx);
      if (r < 8) {
        if (DELTA) sm.Lm[i][j] = sm.beta[i] * acc[e];
      } else {
        sm.Mq[i][j] = p.scale * acc[e];
      }
    }
  }
  __syncthreads();

  {
    typename ST2::T* mq = reinterpret_cast<typename ST2::T*>(rec + R::kMqk);
    for (int e = tid; e < 256; e += kPrepThreads) mq[e] = ST2::cvt(sm.Mq[e >> 4][e & 15]);
  }
  if (!DELTA) return;

  // ---- INV = (I + L)^{-1}, then INV' = INV diag(beta) ----
  if (warp == 0) {
    float* X0 = &sm.X[0][0][0];
    float* X1 = &sm.X[1][0][0];
    float* X2 = &sm.X[2][0][0];
    float* X3 = &sm.X[3][0][0];
    for (int e = lane; e < 256; e += 32) X0[(e >> 4) * 17 + (e & 15)] = -sm.Lm[e >> 4][e & 15];
    __syncwarp();
    warp_mm16<QK>(X0, false, X0, false, X1, lane);  // X^2
    warp_mm16<QK>(X1, false, X1, false, X2, lane);  // X^4
    warp_mm16<QK>(X0, true, X1, true, X3, lane);    // (I+X)(I+X^2)
    warp_mm16<QK>(X2, false, X2, false, X0, lane);  // X^8
    warp_mm16<QK>(X3, false, X2, true, X1, lane);   // ... (I+X^4)
    warp_mm16<QK>(X1, false, X0, true, X3, lane);   // ... (I+X^8) = INV
    for (int e = lane; e < 256; e += 32) {
      const int i = e >> 4, j = e & 15;
      const float v = X3[i * 17 + j] * sm.beta[j];
      sm.invq[i][j] = QK::cvt(v);
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      sm.invhi[i][j] = hi;
      sm.invlo[i][j] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
  }
  __syncthreads();

  // ---- W = INV' k_dec (stored negated) and U~ = INV' v (fp32, transposed) ----
  {
    const int g = lane >> 2, t = lane & 3;
    constexpr int COLS = D / 4;  // columns per warp
    uint32_t a[4], ahi[4], alo[4];
    ldsm_x4(a, &sm.invq[lane & 15][(lane >> 4) * 8]);
    ldsm_x4(ahi, &sm.invhi[lane & 15][(lane >> 4) * 8]);
    ldsm_x4(alo, &sm.invlo[lane & 15][(lane >> 4) * 8]);
    __nv_bfloat16* wneg = reinterpret_cast<__nv_bfloat16*>(rec + R::kW);
    float* ut = reinterpret_cast<float*>(rec + R::kUt);
#pragma unroll
    for (int pp = 0; pp < COLS / 16; ++pp) {
      const int n0 = warp * COLS + 16 * pp;
      uint32_t b[4];
      ldsm_x4_trans(b, &sm.kdec[lane & 15][n0 + (lane >> 4) * 8]);
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816<QK>(c0, a, b[0], b[1]);
      mma16816<QK>(c1, a, b[2], b[3]);
      auto st = [&](int row, int col, float x, float y) {
        *reinterpret_cast<uint32_t*>(wneg + row * D + col) = Bf16::pack(-x, -y);
      };
      st(g, n0 + 2 * t, c0[0], c0[1]);
      st(g + 8, n0 + 2 * t, c0[2], c0[3]);
      st(g, n0 + 8 + 2 * t, c1[0], c1[1]);
      st(g + 8, n0 + 8 + 2 * t, c1[2], c1[3]);

      ldsm_x4_trans(b, &sm.vs[lane & 15][n0 + (lane >> 4) * 8]);
      float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816<Bf16>(u0, ahi, b[0], b[1]);
      mma16816<Bf16>(u0, alo, b[0], b[1]);
      mma16816<Bf16>(u1, ahi, b[2], b[3]);
      mma16816<Bf16>(u1, alo, b[2], b[3]);
      auto su = [&](int tok, int col, float x) { ut[col * 16 + tok] = x; };
      su(g, n0 + 2 * t, u0[0]);
      su(g, n0 + 2 * t + 1, u0[1]);
      su(g + 8, n0 + 2 * t, u0[2]);
      su(g + 8, n0 + 2 * t + 1, u0[3]);
      su(g, n0 + 8 + 2 * t, u1[0]);
      su(g, n0 + 8 + 2 * t + 1, u1[1]);
      su(g + 8, n0 + 8 + 2 * t, u1[2]);
      su(g + 8, n0 + 8 + 2 * t + 1, u1[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// Recurrence
// ---------------------------------------------------------------------------
template <int D, int WARPS, typename S2>
struct RecStage {
  __align__(16) __nv_bfloat16 W[16][D + 8];
  __align__(16) __nv_bfloat16 qd[16][D + 8];
  __align__(16) S2 kr[16][D + 8];
  __align__(16) S2 mqk[16][24];
  __align__(16) float gamma[D];
  __align__(16) float ut[16 * WARPS][16];
};

template <int D, int WARPS, typename S2>
struct RecSmem {
  RecStage<D, WARPS, S2> st[2];
  __align__(16) __nv_bfloat16 ostage[16][16 * WARPS + 8];
};

// PAR = false: the serial chunk recurrence of one (sequence, head, value block),
// writing the state entering every chunk to p.h_chunks when it is given.
// PAR = true: the chunk-parallel output pass: one CTA per (global chunk, head,
// value block) starts from that chunk's entering state in p.h_chunks and forms
// only the chunk's output (the state update is the serial pass's business).
template <int D, int WARPS, bool DELTA, bool PAR>
__global__ void __launch_bounds__(WARPS * 32) kda_recur_tc_kernel(const ChunkCall p) {
  using ST2 = std::conditional_t<DELTA, F16, Bf16>;
  using S2 = typename ST2::T;
  using R = RecTC<D>;
  using Smem = RecSmem<D, WARPS, S2>;
  constexpr int NT = D / 8;  // n-tiles of the state row (key channels)
  constexpr int NTHR = WARPS * 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

  const int H = p.geo.H;
  const int unit = blockIdx.x / H;  // sequence, or global chunk (PAR)
  const int h = blockIdx.x - unit * H;
  const int dv0 = blockIdx.y * 16 * WARPS;
  int n = unit, c_begin = 0;
  if (PAR) {
    ChunkPos pos;
    if (!locate_chunk(p.geo, unit, pos)) return;
    n = pos.n;
    c_begin = pos.c;
  }
  int ts, te, cb;
  if (!locate_seq(p.geo, n, ts, te, cb)) return;
  const int nch = PAR ? c_begin + 1 : (te - ts + kChunk - 1) / kChunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = dv0 + warp * 16;  // first value row of this warp

  float S[NT][4];
  const float* s_src = PAR ? p.h_chunks + (static_cast<size_t>(unit) * H + h) * D * D
                           : (p.h0 != nullptr ? p.h0 + (static_cast<size_t>(n) * H + h) * D * D : nullptr);
  if (s_src != nullptr) {
    const float* src = s_src;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 x = *reinterpret_cast<const float2*>(src + (r0 + g) * D + 8 * nt + 2 * t);
      const float2 y = *reinterpret_cast<const float2*>(src + (r0 + g + 8) * D + 8 * nt + 2 * t);
      S[nt][0] = x.x; S[nt][1] = x.y; S[nt][2] = y.x; S[nt][3] = y.y;
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
  }

  const size_t rec_stride = static_cast<size_t>(H) * R::kBytes;  // between consecutive chunks
  const unsigned char* rec0 = p.records + (static_cast<size_t>(cb) * H + h) * R::kBytes;

  auto load_stage = [&](int c, int si) {
    RecStage<D, WARPS, S2>& st = sm.st[si];
    const unsigned char* rec = rec0 + static_cast<size_t>(c) * rec_stride;
    constexpr int VPR = D / 8;  // 16-byte vectors per 16-bit row
    for (int i = tid; i < 16 * VPR; i += NTHR) {
      const int row = i / VPR, v = i % VPR;
      if (DELTA) cp_async16(&st.W[row][v * 8], rec + R::kW + (row * D + v * 8) * 2);
      cp_async16(&st.qd[row][v * 8], rec + R::kQd + (row * D + v * 8) * 2);
      cp_async16(&st.kr[row][v * 8], rec + R::kKr + (row * D + v * 8) * 2);
    }
    for (int i = tid; i < 32; i += NTHR) cp_async16(&st.mqk[i >> 1][(i & 1) * 8], rec + R::kMqk + i * 16);
    for (int i = tid; i < D / 4; i += NTHR) cp_async16(&st.gamma[i * 4], rec + R::kGamma + i * 16);
    for (int i = tid; i < 16 * WARPS * 4; i += NTHR) {
      const int row = i >> 2, v = i & 3;
      cp_async16(&st.ut[row][v * 4], rec + R::kUt + (static_cast<size_t>(dv0 + row) * 16 + v * 4) * 4);
    }
  };

  if (nch > c_begin) {
    load_stage(c_begin, 0);
    cp_async_commit();
  }
  for (int c = c_begin; c < nch; ++c) {
    const int it = c - c_begin;
    if (c + 1 < nch) {
      load_stage(c + 1, (it + 1) & 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const RecStage<D, WARPS, S2>& st = sm.st[it & 1];
    if (!PAR && p.h_chunks != nullptr) {  // the state entering chunk c
      float* dst = p.h_chunks + (static_cast<size_t>(cb + c) * H + h) * D * D;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        *reinterpret_cast<float2*>(dst + (r0 + g) * D + 8 * nt + 2 * t) = make_float2(S[nt][0], S[nt][1]);
        *reinterpret_cast<float2*>(dst + (r0 + g + 8) * D + 8 * nt + 2 * t) = make_float2(S[nt][2], S[nt][3]);
      }
    }

    // S^T as bf16 A fragments (accumulator layout == A layout for tile pairs)
    uint32_t sa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      sa[kk][0] = Bf16::pack(S[2 * kk][0], S[2 * kk][1]);
      sa[kk][1] = Bf16::pack(S[2 * kk][2], S[2 * kk][3]);
      sa[kk][2] = Bf16::pack(S[2 * kk + 1][0], S[2 * kk + 1][1]);
      sa[kk][3] = Bf16::pack(S[2 * kk + 1][2], S[2 * kk + 1][3]);
    }
    float u[2][4], u2[2][4], o[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float2 x = *reinterpret_cast<const float2*>(&st.ut[warp * 16 + g][8 * nt + 2 * t]);
      const float2 y = *reinterpret_cast<const float2*>(&st.ut[warp * 16 + g + 8][8 * nt + 2 * t]);
      u[nt][0] = x.x; u[nt][1] = x.y; u[nt][2] = y.x; u[nt][3] = y.y;
#pragma unroll
      for (int e = 0; e < 4; ++e) { u2[nt][e] = 0.f; o[nt][e] = 0.f; }
    }
    // stage 1: U^T += S^T (-W)^T ; O^T = S^T q_dec^T
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int row = ((lane >> 4) << 3) + (lane & 7);
      const int col = 16 * kk + ((lane >> 3) & 1) * 8;
      uint32_t b[4];
      if (DELTA) {
        ldsm_x4(b, &st.W[row][col]);
        float (&acc)[2][4] = (kk & 1) ? u2 : u;
        mma16816<Bf16>(acc[0], sa[kk], b[0], b[1]);
        mma16816<Bf16>(acc[1], sa[kk], b[2], b[3]);
      }
      ldsm_x4(b, &st.qd[row][col]);
      mma16816<Bf16>(o[0], sa[kk], b[0], b[1]);
      mma16816<Bf16>(o[1], sa[kk], b[2], b[3]);
    }
    uint32_t ua[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) u[nt][e] += u2[nt][e];
    ua[0] = ST2::pack(u[0][0], u[0][1]);
    ua[1] = ST2::pack(u[0][2], u[0][3]);
    ua[2] = ST2::pack(u[1][0], u[1][1]);
    ua[3] = ST2::pack(u[1][2], u[1][3]);

    // stage 2a: S^T = S^T diag(gamma) + U^T k_res   (the serial dependency)
#pragma unroll
    for (int np = 0; np < (PAR ? 0 : D / 16); ++np) {
      uint32_t b[4];
      ldsm_x4_trans(b, &st.kr[lane & 15][16 * np + (lane >> 4) * 8]);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int nt = 2 * np + half;
        const float2 gm = *reinterpret_cast<const float2*>(&st.gamma[8 * nt + 2 * t]);
        S[nt][0] *= gm.x; S[nt][1] *= gm.y; S[nt][2] *= gm.x; S[nt][3] *= gm.y;
        mma16816<ST2>(S[nt], ua, b[2 * half], b[2 * half + 1]);
      }
    }
    // stage 2b: O^T += U^T Mqk^T
    {
      uint32_t b[4];
      const int row = ((lane >> 4) << 3) + (lane & 7);
      ldsm_x4(b, &st.mqk[row][((lane >> 3) & 1) * 8]);
      mma16816<ST2>(o[0], ua, b[0], b[1]);
      mma16816<ST2>(o[1], ua, b[2], b[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tok = 8 * nt + 2 * t;
      sm.ostage[tok][warp * 16 + g] = __float2bfloat16_rn(o[nt][0]);
      sm.ostage[tok + 1][warp * 16 + g] = __float2bfloat16_rn(o[nt][1]);
      sm.ostage[tok][warp * 16 + g + 8] = __float2bfloat16_rn(o[nt][2]);
      sm.ostage[tok + 1][warp * 16 + g + 8] = __float2bfloat16_rn(o[nt][3]);
    }
    __syncthreads();
    {
      constexpr int VPR = 2 * WARPS;  // 16-byte vectors per token row of this CTA
      const int tok0 = ts + c * kChunk;
      const int ntok = min(kChunk, te - tok0);
      for (int i = tid; i < 16 * VPR; i += NTHR) {
        const int row = i / VPR, v = i % VPR;
        if (row < ntok) {
          __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) +
                               (static_cast<size_t>(tok0 + row) * H + h) * D + dv0 + v * 8;
          *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&sm.ostage[row][v * 8]);
        }
      }
    }
  }

  if (!PAR && p.hT != nullptr) {
    float* dst = p.hT + (static_cast<size_t>(n) * H + h) * D * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(dst + (r0 + g) * D + 8 * nt + 2 * t) = make_float2(S[nt][0], S[nt][1]);
      *reinterpret_cast<float2*>(dst + (r0 + g + 8) * D + 8 * nt + 2 * t) = make_float2(S[nt][2], S[nt][3]);
    }
  }
}

template <int D, bool DELTA, bool L2N>
cudaError_t launch_prep_t(const ChunkCall& c, cudaStream_t s) {
  if (c.geo.max_chunks == 0) return cudaSuccess;
  dim3 grid(c.geo.max_chunks, c.geo.H);
  kda_prep_tc_kernel<D, DELTA, L2N><<<grid, kPrepThreads, 0, s>>>(c);
  return cudaGetLastError();
}

template <int D, bool DELTA, bool PAR>
cudaError_t launch_recur_t(const ChunkCall& c, cudaStream_t s) {
  constexpr int WARPS = 2;
  using ST2 = std::conditional_t<DELTA, F16, Bf16>;
  using Smem = RecSmem<D, WARPS, typename ST2::T>;
  const size_t smem = sizeof(Smem);
  static std::atomic<uint64_t> smem_set{0};  // per instantiation and device
  {
    const cudaError_t e = set_smem_limit_once(kda_recur_tc_kernel<D, WARPS, DELTA, PAR>, smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  const unsigned units = PAR ? static_cast<unsigned>(c.geo.max_chunks) : static_cast<unsigned>(c.geo.N);
  if (units == 0) return cudaSuccess;
  dim3 grid(units * c.geo.H, D / (16 * WARPS));
  kda_recur_tc_kernel<D, WARPS, DELTA, PAR><<<grid, WARPS * 32, smem, s>>>(c);
  return cudaGetLastError();
}

template <int D, bool PAR>
cudaError_t launch_chunk_tc_d(const ChunkCall& c, cudaStream_t s) {
  cudaError_t e;
  if (c.delta) {
    e = c.l2norm ? launch_prep_t<D, true, true>(c, s) : launch_prep_t<D, true, false>(c, s);
    if (e != cudaSuccess) return e;
    return launch_recur_t<D, true, PAR>(c, s);
  }
  e = c.l2norm ? launch_prep_t<D, false, true>(c, s) : launch_prep_t<D, false, false>(c, s);
  if (e != cudaSuccess) return e;
  return launch_recur_t<D, false, PAR>(c, s);
}

}  // namespace

size_t record_bytes_tc(int d) {
  if (d == 128) return RecTC<128>::kBytes;
  if (d == 64) return RecTC<64>::kBytes;
  return 0;
}

cudaError_t launch_chunk_tc(const ChunkCall& c, cudaStream_t s) {
  if (c.dk == 128) return launch_chunk_tc_d<128, false>(c, s);
  if (c.dk == 64) return launch_chunk_tc_d<64, false>(c, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_output_tc(const ChunkCall& c, cudaStream_t s) {
  if (c.h_chunks == nullptr) return cudaErrorInvalidValue;
  if (c.dk == 128) return launch_chunk_tc_d<128, true>(c, s);
  if (c.dk == 64) return launch_chunk_tc_d<64, true>(c, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
