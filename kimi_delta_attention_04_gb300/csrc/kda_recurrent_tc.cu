// Short-T KDA recurrent step on a state-slot pool, on the tensor cores.
//
// The operation is that of kda_recurrent.cu (the general fused recurrent path
// that the packed decode specialises; sglang PR #26586 summary, 功能与动机 and
// 实现拆解): T <= 64 tokens per batch row applied in order to the row's slot,
// separate q/k/v tensors, value-head grouping hv -> hv / (HV / H), q and k
// L2-normalised (eps 1e-6 in the root), g = -exp(A_log) softplus(a + dt_bias)
// per key channel, beta = sigmoid(b).
//
// GB300 design. The T tokens of a row are ceil(T/16) chunks of the chunkwise
// form ("FlashKDA里的L矩阵和Mqk矩阵": L, Mqk, the Neumann inverse, the chunk step
// "U = INV beta (v - k_dec S); out = q_dec S + Mqk U; S = e^{g_total} S +
// k_res^T U"), so the state work runs as mma.sync m16n8k16 with fp32
// accumulation instead of per-token FMA loops. One CTA of 4 warps per
// (row, value head), four CTAs per SM:
//  * the CTA first asks L2 for the row's 64 KiB slot (bulk prefetch), stages
//    the chunk's q, k, a and v rows with 16-byte cp.async, then prepares the
//    chunk with one thread per key channel (L2 norms, decay products, the
//    anchored level split of L and Mqk into channel-major tiles, each warp
//    forming the inverse in registers for its columns of W and U~);
//  * each warp owns V / 4 value rows of the state and steps them 16 at a
//    time, S^T [16 x K] fp32 in registers as MMA accumulators, loaded after
//    the chunk's preparation and stored back after its step: U^T = U~^T -
//    S^T W^T, O^T = S^T q_dec^T + U^T Mqk^T, S^T = S^T diag(gamma) + U^T k_res.
//    The slot is read before the first chunk and written after the last; in
//    between, with d_k = 128, a row of more than 16 tokens keeps its state tiles
//    in tensor memory (tcgen05.st / tcgen05.ld: each warp its own lane quarter,
//    MT * 64 columns per CTA, so four CTAs fill at most an SM's 512 columns)
//    instead of an L2 round trip per chunk, which at 64 tokens per row made ~40 %
//    of the L1 data-pipe wavefronts (16-byte state accesses, each warp access
//    touching eight half-used lines);
//  * o is staged in shared memory and written as 16-byte rows.
// Operand precision as in the chunk forward: S, W, q_dec bf16; U, k_res, Mqk
// fp16; L/Mqk/INV operands fp16 (q, k normalised) or bf16; U~ fp32.
#include <type_traits>

#include "kda_cluster.cuh"
#include "kda_common.cuh"
#include "kda_tcgen05.cuh"

namespace kda {
namespace {

constexpr int kMaxT = 64;

constexpr size_t rt_max(size_t x, size_t y) { return x > y ? x : y; }

// Shared memory of one CTA. Three buffers live one after another in `region`:
// the chunk's staged inputs (until each thread has read its channel), the level
// operands (until the L / Mqk MMAs), then -W, U~^T and the output staging
// (through the step). Barriers separate the phases, so the CTA needs ~48 KB
// (K = V = 128) and four fit on an SM.
template <int K, int V, typename Q>
struct RtcSmem {
  struct In {  // [token][channel], rows past T zeroed
    __nv_bfloat16 q[16][K];
    __nv_bfloat16 k[16][K];
    __nv_bfloat16 a[16][K];
    __nv_bfloat16 v[16][V];
  };
  struct Lv {
    Q A[4][K][16];  // per level, channel-major: rows 0-7 k*F, rows 8-15 q*F of the row tokens
    Q B[4][K][8];   // per level, channel-major: k*F of the column tokens
  };
  struct St {
    __nv_bfloat16 W[16][K + 8];  // -W = -(INV diag(beta) k_dec), [token][channel]
    float ut[V][24];             // U~^T [value row][token]
    __nv_bfloat16 ostage[16][V + 8];
  };
  __align__(16) unsigned char region[rt_max(sizeof(In), rt_max(sizeof(Lv), sizeof(St)))];
  // channel-major [channel][16 tokens] tiles (halves swizzled, rt_cm_off)
  __align__(16) Q kdec[K][16];
  __align__(16) __nv_bfloat16 vs[V][16];
  __align__(16) __nv_bfloat16 qd[K][16];  // scale q e^{G}
  __align__(16) __half kr[K][16];         // k e^{G_last - G}
  __align__(16) __half mqk[16][24];
  __align__(16) float gamma[K];
  float Lm[16][17];
  float Mq[16][17];
  float red[K / 32][48];
  float rnq[16], rnk[16], beta[16];
  uint32_t tmem_base;  // tensor-memory columns holding the state between chunks (rows of > 16 tokens)
  __device__ __forceinline__ In& in() { return *reinterpret_cast<In*>(region); }
  __device__ __forceinline__ Lv& lv() { return *reinterpret_cast<Lv*>(region); }
  __device__ __forceinline__ St& st() { return *reinterpret_cast<St*>(region); }
};

// Channel-major 16-bit tiles [channel][16 tokens]: a channel's 16 tokens are one
// 32-byte row, written by the thread that owns the channel with two 16-byte
// stores; the two halves (tokens 0-7, 8-15) are swapped on rows whose bits 2 and 3
// differ. The eight rows of one ldmatrix 8x8 load (bit 3 fixed) fall on distinct
// banks, and so do the rows eight consecutive channels write, both in channel
// order and in the MMAs' key order (rt_mma_key), where they are rows
// {0, 1, 8, 9, 2, 3, 10, 11} (+ 4) of a 16-row block.
__device__ __forceinline__ int rt_cm_off(int row, int half) {
  return row * 16 + ((half ^ (row >> 2) ^ (row >> 3)) & 1) * 8;
}

// Column of U~^T [value row][token] in shared memory. With SWZ = 8 the token index is
// XORed with 8 on rows whose bit 2 is set, so the scalar stores of one MMA fragment
// (rows 2 t apart, columns g) are conflict-free as well as the float2 loads of the step
// (rows g, columns 2 t). The d_k = 64 instances keep the plain layout (SWZ = 0): one of
// them has no register to spare for the extra index arithmetic.
template <int SWZ>
__device__ __forceinline__ int rt_ut_col(int row, int tok) { return tok ^ (((row >> 2) & 1) * SWZ); }

// Key order inside the state step. Within each block of 16 keys, the key the
// MMAs call 8 j + 2 t + e (n-tile j of the pair, accumulator column pair of lane
// t) is stored key 4 t + 2 j + e, so the four keys a lane holds across the pair
// are consecutive in memory and the state moves between L2 and registers as one
// 16-byte access per row and pair of n-tiles. The operands indexed by key
// (q_dec, k_res, k_dec) are laid out in the MMAs' order and gamma by stored key (a
// lane's four decay factors of a pair of n-tiles are one 16-byte load); L and Mqk sum
// over every key and do not care.
__device__ __forceinline__ int rt_mma_key(int key) {
  const int r = key & 15;
  return (key & ~15) + ((r >> 1) & 1) * 8 + (r >> 2) * 2 + (r & 1);
}

// Token of row r (column r) of a level's 8-row block, the level's half-block size
// being s = 2^ls (shifts: the level is a warp index, so a division would be a
// run-time one).
__device__ __forceinline__ int rt_row_tok(int ls, int r) { return ((r >> ls) << (ls + 1)) + (1 << ls) + (r & ((1 << ls) - 1)); }
__device__ __forceinline__ int rt_col_tok(int ls, int r) { return ((r >> ls) << (ls + 1)) + (r & ((1 << ls) - 1)); }

// RES: the state stays in tensor memory between chunks (d_k = 128, T > 16). Rows of
// one chunk launch the instance without it, which holds no tcgen05 instruction: a CTA
// of a kernel that allocates tensor memory keeps the SM's allocation permit until it
// relinquishes it or exits, and at 8 tokens per row the allocating instance ran at
// half speed even where it allocated nothing (185 vs 98 us at 128 rows; relinquishing
// at the start of every CTA took it back to 101 us).
template <int K, int V, bool L2N, bool RES>
__global__ void __launch_bounds__(128, 4) kda_recurrent_tc_kernel(const RecurrentCall p) {
  using QK = std::conditional_t<L2N, F16, Bf16>;
  using Q = typename QK::T;
  constexpr int WARPS = 4;
  constexpr int NTHR = 32 * WARPS;
  constexpr int MT = V / (16 * WARPS);  // 16-row tiles of the state per warp
  constexpr int NT = K / 8;             // n-tiles of a state row
  constexpr int KK = K / 16;            // k-steps over the key channels
  constexpr int kUtSwz = K == 128 ? 8 : 0;  // column swizzle of U~^T (rt_ut_col)
  static_assert(NTHR >= K && NTHR >= V, "one thread per key and per value channel");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  using Smem = RtcSmem<K, V, Q>;
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  typename Smem::In& in = sm.in();
  typename Smem::Lv& lvo = sm.lv();
  typename Smem::St& st = sm.st();

  const int T = p.T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int unit = blockIdx.x;  // b * HV + hv
  const int b = unit / p.HV;
  const int hv = unit - b * p.HV;
  const int h = hv / (p.HV / p.H);
  const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(p.v);
  const __nv_bfloat16* ab = reinterpret_cast<const __nv_bfloat16*>(p.a);
  const __nv_bfloat16* bb = reinterpret_cast<const __nv_bfloat16*>(p.b);

  const int slot = p.indices[b];
  if (slot < 0 || slot >= p.num_slots) {
    if (slot >= p.num_slots && tid == 0) set_err(p.err, 1 /* KDA_ERR_INVALID_ARG */);
    for (int i = tid; i < T * (V / 8); i += NTHR) {
      const int tok = i / (V / 8), v8 = i - tok * (V / 8);
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                ((static_cast<size_t>(b) * T + tok) * p.HV + hv) * V + v8 * 8) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  float* const S_slot = p.state_pool + (static_cast<size_t>(slot) * p.HV + hv) * static_cast<size_t>(V) * K;
  if (tid == 0) {
    constexpr uint32_t kPart = 16384;
    for (uint32_t off = 0; off < static_cast<uint32_t>(V * K * 4); off += kPart)
      bulk_prefetch_l2(reinterpret_cast<const unsigned char*>(S_slot) + off, kPart);
  }

  const bool kown = tid < K;
  const bool vown = tid < V;
  const int ch = kown ? tid : 0;
  const float Aexp = expf(p.A_log[hv]);
  const float dtb = kown ? p.dt_bias[hv * K + ch] : 0.f;

  const int nch = (T + 15) / 16;
  // Tensor memory for the state between chunks (d_k = 128 only: at d_k = 64 the
  // round trip is half as large and that instance has no registers to spare for
  // it). Occupancy is at most four CTAs per SM (registers), so the columns are
  // there (a fifth CTA would only wait in the allocation until another one exits);
  // every CTA that allocates reaches the release after the chunk loop (no return
  // in between).
  static_assert(!RES || K == 128, "tensor-memory state at d_k = 128 only");
  constexpr bool kTmemState = RES;
  constexpr int kTileCols = NT * 4;  // one 16-row tile: 64 fp32 accumulators per lane
  constexpr uint32_t kTmemCols = MT * kTileCols;
  static_assert(!kTmemState || (kTmemCols >= 32 && kTmemCols <= 128 && (kTmemCols & (kTmemCols - 1)) == 0),
                "a power of two of at most 512 / 4 columns");
  const bool resident = kTmemState && nch > 1;  // (the launcher takes RES only for T > 16)
  uint32_t tbase = 0;
  if (resident) {
    if (warp == 0) {
      tc05::tmem_alloc(&sm.tmem_base, kTmemCols);
      tc05::tmem_relinquish();
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    tbase = sm.tmem_base + (static_cast<uint32_t>(32 * warp) << 16);  // this warp's lane quarter
  }
  for (int c = 0; c < nch; ++c) {
    const int tok0 = 16 * c;
    const int ntok = min(16, T - tok0);
    // ---------------- chunk preparation ----------------
    {  // 16-byte rows of q, k (head h), a and v (value head hv)
      const size_t bt0 = static_cast<size_t>(b) * T + tok0;
      for (int i = tid; i < 16 * (K / 8); i += NTHR) {
        const int row = i / (K / 8), c8 = i - row * (K / 8);
        if (row < ntok) {
          const size_t qk = ((bt0 + row) * p.H + h) * K + c8 * 8;
          cp_async16(&in.q[row][c8 * 8], qb + qk);
          cp_async16(&in.k[row][c8 * 8], kb + qk);
          cp_async16(&in.a[row][c8 * 8], ab + ((bt0 + row) * p.HV + hv) * K + c8 * 8);
        } else {
          *reinterpret_cast<uint4*>(&in.q[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(&in.k[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(&in.a[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
        }
      }
      for (int i = tid; i < 16 * (V / 8); i += NTHR) {
        const int row = i / (V / 8), c8 = i - row * (V / 8);
        if (row < ntok) cp_async16(&in.v[row][c8 * 8], vb + ((bt0 + row) * p.HV + hv) * V + c8 * 8);
        else *reinterpret_cast<uint4*>(&in.v[row][c8 * 8]) = make_uint4(0, 0, 0, 0);
      }
      cp_async_commit();
    }
    for (int i = tid; i < 16 * 17; i += NTHR) {
      (&sm.Lm[0][0])[i] = 0.f;
      (&sm.Mq[0][0])[i] = 0.f;
    }
    if (tid < 16) {
      float bt = 0.f;
      if (tid < ntok) bt = sigmoid_f(__bfloat162float(bb[(static_cast<size_t>(b) * T + tok0 + tid) * p.HV + hv]));
      sm.beta[tid] = bt;
    }
    cp_async_wait<0>();
    __syncthreads();
    float qv[16], kv[16], al[16];
    if (kown) {
      constexpr float kLog2e = 1.4426950408889634f;
      const float nA = -Aexp;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool valid = i < ntok;
        qv[i] = __bfloat162float(in.q[i][ch]);
        kv[i] = __bfloat162float(in.k[i][ch]);
        const float x = __bfloat162float(in.a[i][ch]) + dtb;
        // alpha = e^{-A softplus(x)} = 2^{-A log2(1 + 2^{x log2 e})}, x itself above 20
        const float l2 = lg2_approx(1.f + ex2_approx(fminf(x, 20.f) * kLog2e));
        const float sp2 = x > 20.f ? x * kLog2e : l2;
        al[i] = valid ? ex2_approx(nA * sp2) : 1.f;
      }
      // this warp's partial sums of q.q, k.k and q.k per token over its 32 channels:
      // the diagonals of Q Q^T, K K^T and Q K^T on the tensor cores (bf16 products
      // are exact in fp32), from raw channel-major rows staged in the q_dec and
      // k_dec tiles (written again only after the next two barriers); as A
      // operands [token][channel] they come from .trans loads, and the B fragments
      // of Q^T (K^T) are the A fragments of Q (K) in another order
      uint16_t* const rq_t = reinterpret_cast<uint16_t*>(&sm.qd[0][0]);
      uint16_t* const rk_t = reinterpret_cast<uint16_t*>(&sm.kdec[0][0]);
      {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = Bf16::pack(qv[2 * i], qv[2 * i + 1]);
        *reinterpret_cast<uint4*>(rq_t + rt_cm_off(ch, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(rq_t + rt_cm_off(ch, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = Bf16::pack(kv[2 * i], kv[2 * i + 1]);
        *reinterpret_cast<uint4*>(rk_t + rt_cm_off(ch, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(rk_t + rt_cm_off(ch, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      __syncwarp();
      {
        // lane matrix m of an A fragment: (channel half m >> 1, token half m & 1)
        const int r_row = ((lane >> 4) & 1) * 8 + (lane & 7), r_half = (lane >> 3) & 1;
        float dqq[2][4] = {}, dkk[2][4] = {}, dqk[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t aq[4], ak[4];
          ldsm_x4_trans(aq, rq_t + rt_cm_off(32 * warp + 16 * ks + r_row, r_half));
          ldsm_x4_trans(ak, rk_t + rt_cm_off(32 * warp + 16 * ks + r_row, r_half));
          mma16816<Bf16>(dqq[0], aq, aq[0], aq[2]);
          mma16816<Bf16>(dqq[1], aq, aq[1], aq[3]);
          mma16816<Bf16>(dkk[0], ak, ak[0], ak[2]);
          mma16816<Bf16>(dkk[1], ak, ak[1], ak[3]);
          mma16816<Bf16>(dqk[0], aq, ak[0], ak[2]);
          mma16816<Bf16>(dqk[1], aq, ak[1], ak[3]);
        }
        // diagonal element (i, i): token tile i / 8, lane (i % 8, (i % 8) / 2),
        // entry (i % 8) % 2 (+2 in the second token tile)
        if ((g >> 1) == t) {
          const int e = g & 1;
          sm.red[warp][g] = e ? dqq[0][1] : dqq[0][0];
          sm.red[warp][8 + g] = e ? dqq[1][3] : dqq[1][2];
          sm.red[warp][16 + g] = e ? dkk[0][1] : dkk[0][0];
          sm.red[warp][24 + g] = e ? dkk[1][3] : dkk[1][2];
          sm.red[warp][32 + g] = e ? dqk[0][1] : dqk[0][0];
          sm.red[warp][40 + g] = e ? dqk[1][3] : dqk[1][2];
        }
      }
    }
    if (vown) {  // v rows into the channel-major tile (raw bf16 bits, two tokens per word)
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = static_cast<uint32_t>(__bfloat16_as_ushort(in.v[2 * i][tid])) |
               (static_cast<uint32_t>(__bfloat16_as_ushort(in.v[2 * i + 1][tid])) << 16);
      uint16_t* tile = reinterpret_cast<uint16_t*>(&sm.vs[0][0]);
      *reinterpret_cast<uint4*>(tile + rt_cm_off(tid, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(tile + rt_cm_off(tid, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    __syncthreads();
    if (tid < 16) {
      float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
      for (int w = 0; w < K / 32; ++w) {
        sq += sm.red[w][tid];
        sk += sm.red[w][16 + tid];
        sqk += sm.red[w][32 + tid];
      }
      const float rq = p.l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
      const float rk = p.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
      sm.rnq[tid] = rq;
      sm.rnk[tid] = rk;
      sm.Mq[tid][tid] = p.scale * sqk * rq * rk;
    }
    __syncthreads();
    if (kown) {
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
      // channel ch's 16 tokens of each channel-major tile, two 16-byte stores each
      const int mk = rt_mma_key(ch);  // this channel's row in the key-indexed operand tiles
      auto put16 = [&](void* tile, const uint32_t (&w)[8]) {
        uint16_t* base = reinterpret_cast<uint16_t*>(tile);
        *reinterpret_cast<uint4*>(base + rt_cm_off(mk, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(base + rt_cm_off(mk, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
      };
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = Bf16::pack(p.scale * qv[2 * i] * P[2 * i], p.scale * qv[2 * i + 1] * P[2 * i + 1]);
      put16(&sm.qd[0][0], w);
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = F16::pack(kv[2 * i] * Rs[2 * i], kv[2 * i + 1] * Rs[2 * i + 1]);
      put16(&sm.kr[0][0], w);
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = QK::pack(kv[2 * i] * P[2 * i], kv[2 * i + 1] * P[2 * i + 1]);
      put16(&sm.kdec[0][0], w);
      sm.gamma[ch] = P[15];
#pragma unroll
      for (int lv = 0; lv < 4; ++lv) {
        const int s = 8 >> lv;
        float ar[16], bc[8];  // this channel's row (k rows 0-7, q rows 8-15) and column operands
#pragma unroll
        for (int blk = 0; blk < 8 / s; ++blk) {
          const int m = blk * 2 * s + s;  // anchor: first row of the upper half
          float f = 1.f;
#pragma unroll
          for (int i = m; i < m + s; ++i) {  // row tokens: prod_{m<t<=i} alpha_t
            if (i > m) f *= al[i];
            const int r = blk * s + (i - m);
            ar[r] = kv[i] * f;
            ar[8 + r] = qv[i] * f;
          }
          f = 1.f;
#pragma unroll
          for (int i = m - 1; i >= m - s; --i) {  // column tokens: prod_{i<t<=m} alpha_t
            f *= al[i + 1];
            bc[blk * s + (i - (m - s))] = kv[i] * f;
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = QK::pack(ar[2 * i], ar[2 * i + 1]);
        {  // the level tiles are summed over every channel: physical order
          uint16_t* base = reinterpret_cast<uint16_t*>(&lvo.A[lv][0][0]);
          *reinterpret_cast<uint4*>(base + rt_cm_off(ch, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(base + rt_cm_off(ch, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        *reinterpret_cast<uint4*>(&lvo.B[lv][ch][0]) =
            make_uint4(QK::pack(bc[0], bc[1]), QK::pack(bc[2], bc[3]), QK::pack(bc[4], bc[5]), QK::pack(bc[6], bc[7]));
      }
    }
    __syncthreads();
    if (warp < 4) {  // level `warp` of the anchored split: L (rows 0-7) and Mqk (rows 8-15)
      const int lv = warp;
      const int ls = 3 - lv;  // half-block size 2^ls = 8 >> lv
      // two accumulator chains, operands loaded one step ahead (mma.sync and
      // ldmatrix keep their program order). A and B are stored [channel][row]:
      // .trans loads; lane matrix m of A = (row half m & 1, channel half m >> 1)
      float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int a_row = (lane >> 4) * 8 + (lane & 7), a_half = (lane >> 3) & 1;
      uint32_t a[2][4], bq[2][2];
      ldsm_x4_trans(a[0], &lvo.A[lv][0][0] + rt_cm_off(a_row, a_half));
      ldsm_x2_trans(bq[0], &lvo.B[lv][lane & 15][0]);
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
        const int cur = kk & 1;
        if (kk + 1 < KK) {
          ldsm_x4_trans(a[cur ^ 1], &lvo.A[lv][0][0] + rt_cm_off(16 * (kk + 1) + a_row, a_half));
          ldsm_x2_trans(bq[cur ^ 1], &lvo.B[lv][16 * (kk + 1) + (lane & 15)][0]);
        }
        mma16816<QK>(acc2[cur], a[cur], bq[cur][0], bq[cur][1]);
      }
      float acc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = acc2[0][e] + acc2[1][e];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g + ((e & 2) ? 8 : 0);
        const int cidx = 2 * t + (e & 1);
        const int rr = r & 7;
        if ((rr >> ls) != (cidx >> ls)) continue;  // not a pair of this level
        const int i = rt_row_tok(ls, rr), j = rt_col_tok(ls, cidx);
        if (r < 8) sm.Lm[i][j] = sm.beta[i] * acc[e];
        else sm.Mq[i][j] = p.scale * acc[e];
      }
    }
    __syncthreads();
    for (int e = tid; e < 256; e += NTHR) sm.mqk[e >> 4][e & 15] = __float2half_rn(sm.Mq[e >> 4][e & 15]);
    {
      // INV' = (I + L)^{-1} diag(beta), formed by every warp in registers
      Frag16 inv = neumann_inverse16<QK>(&sm.Lm[0][0], 17, lane);
      Frag16 ihi, ilo;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = inv.c[nt][e] * sm.beta[8 * nt + 2 * t + (e & 1)];
          inv.c[nt][e] = x;
          ihi.c[nt][e] = __bfloat162float(__float2bfloat16_rn(x));
          ilo.c[nt][e] = x - ihi.c[nt][e];
        }
      uint32_t a[4], ahi[4], alo[4];
      frag_as_a<QK>(inv, a);
      frag_as_a<Bf16>(ihi, ahi);
      frag_as_a<Bf16>(ilo, alo);
      for (int blk = warp; blk < K / 16; blk += WARPS) {  // -W, 16 key channels per block
        const int n0 = 16 * blk;
        uint32_t bw[4];
        ldsm_x4(bw, &sm.kdec[0][0] + rt_cm_off(n0 + (lane >> 4) * 8 + (lane & 7), (lane >> 3) & 1));
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816<QK>(c0, a, bw[0], bw[1]);
        mma16816<QK>(c1, a, bw[2], bw[3]);
        *reinterpret_cast<uint32_t*>(&st.W[g][n0 + 2 * t]) = Bf16::pack(-c0[0], -c0[1]);
        *reinterpret_cast<uint32_t*>(&st.W[g + 8][n0 + 2 * t]) = Bf16::pack(-c0[2], -c0[3]);
        *reinterpret_cast<uint32_t*>(&st.W[g][n0 + 8 + 2 * t]) = Bf16::pack(-c1[0], -c1[1]);
        *reinterpret_cast<uint32_t*>(&st.W[g + 8][n0 + 8 + 2 * t]) = Bf16::pack(-c1[2], -c1[3]);
      }
      for (int blk = warp; blk < V / 16; blk += WARPS) {  // U~ (fp32 through a hi/lo split), 16 value channels
        const int n0 = 16 * blk;
        uint32_t bv[4];
        ldsm_x4(bv, &sm.vs[0][0] + rt_cm_off(n0 + (lane >> 4) * 8 + (lane & 7), (lane >> 3) & 1));
        float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816<Bf16>(u0, ahi, bv[0], bv[1]);
        mma16816<Bf16>(u0, alo, bv[0], bv[1]);
        mma16816<Bf16>(u1, ahi, bv[2], bv[3]);
        mma16816<Bf16>(u1, alo, bv[2], bv[3]);
        st.ut[n0 + 2 * t][rt_ut_col<kUtSwz>(n0 + 2 * t, g)] = u0[0];
        st.ut[n0 + 2 * t + 1][rt_ut_col<kUtSwz>(n0 + 2 * t + 1, g)] = u0[1];
        st.ut[n0 + 2 * t][rt_ut_col<kUtSwz>(n0 + 2 * t, g + 8)] = u0[2];
        st.ut[n0 + 2 * t + 1][rt_ut_col<kUtSwz>(n0 + 2 * t + 1, g + 8)] = u0[3];
        st.ut[n0 + 8 + 2 * t][rt_ut_col<kUtSwz>(n0 + 8 + 2 * t, g)] = u1[0];
        st.ut[n0 + 8 + 2 * t + 1][rt_ut_col<kUtSwz>(n0 + 8 + 2 * t + 1, g)] = u1[1];
        st.ut[n0 + 8 + 2 * t][rt_ut_col<kUtSwz>(n0 + 8 + 2 * t, g + 8)] = u1[2];
        st.ut[n0 + 8 + 2 * t + 1][rt_ut_col<kUtSwz>(n0 + 8 + 2 * t + 1, g + 8)] = u1[3];
      }
    }
    __syncthreads();

    // ---------------- chunk step, one 16-row tile of the state at a time ----------------
#pragma unroll 1
    for (int mt = 0; mt < MT; ++mt) {
      const int r0 = (warp + WARPS * mt) * 16;  // first value row of the tile
      float S[NT][4];
      const uint32_t taddr = tbase + static_cast<uint32_t>(mt * kTileCols);
      // (S as one array of kTileCols floats: column 4 j + e of the tile holds S[j][e])
      float (&s_cols)[kTileCols] = *reinterpret_cast<float(*)[kTileCols]>(&S[0][0]);
      if (kTmemState && c > 0) {  // the tile as this warp left it after the previous chunk
        if constexpr (kTmemState) tc05::ld64_wait(taddr, s_cols);
      } else {  // from the slot, in the accumulator layout (its lines are in L2 by now): stored
                // keys 16 pp + 4 t .. + 3 are MMA keys 16 pp + 2 t (+1) and 16 pp + 8 + 2 t (+1)
#pragma unroll
        for (int pp = 0; pp < NT / 2; ++pp) {
          const float4 x = __ldcs(reinterpret_cast<const float4*>(S_slot + (r0 + g) * K + 16 * pp + 4 * t));
          const float4 y = __ldcs(reinterpret_cast<const float4*>(S_slot + (r0 + g + 8) * K + 16 * pp + 4 * t));
          S[2 * pp][0] = x.x; S[2 * pp][1] = x.y; S[2 * pp + 1][0] = x.z; S[2 * pp + 1][1] = x.w;
          S[2 * pp][2] = y.x; S[2 * pp][3] = y.y; S[2 * pp + 1][2] = y.z; S[2 * pp + 1][3] = y.w;
        }
      }

      float u[2][4], u2[2][4], o[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float2 x = *reinterpret_cast<const float2*>(&st.ut[r0 + g][rt_ut_col<kUtSwz>(r0 + g, 8 * nt + 2 * t)]);
        const float2 y = *reinterpret_cast<const float2*>(&st.ut[r0 + g + 8][rt_ut_col<kUtSwz>(r0 + g + 8, 8 * nt + 2 * t)]);
        u[nt][0] = x.x; u[nt][1] = x.y; u[nt][2] = y.x; u[nt][3] = y.y;
#pragma unroll
        for (int e = 0; e < 4; ++e) { u2[nt][e] = 0.f; o[nt][e] = 0.f; }
      }
      // U^T = U~^T + S^T (-W)^T ; O^T = S^T q_dec^T (S^T as bf16 A fragments, one
      // k-step at a time: the accumulator layout of two n-tiles is the A layout).
      // mma.sync and ldmatrix keep their program order, so each k-step's operands
      // are loaded one step ahead of their MMAs.
      const int w_row = ((lane >> 4) << 3) + (lane & 7), w_col = ((lane >> 3) & 1) * 8;
      const int q_row = ((lane >> 3) & 1) * 8 + (lane & 7), q_half = lane >> 4;
      uint32_t bw[2][4], bqd[2][4];
      ldsm_x4(bw[0], &st.W[w_row][w_col]);
      ldsm_x4_trans(bqd[0], &sm.qd[0][0] + rt_cm_off(q_row, q_half));
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
        const int cur = kk & 1;
        if (kk + 1 < KK) {
          ldsm_x4(bw[cur ^ 1], &st.W[w_row][16 * (kk + 1) + w_col]);
          ldsm_x4_trans(bqd[cur ^ 1], &sm.qd[0][0] + rt_cm_off(16 * (kk + 1) + q_row, q_half));
        }
        uint32_t sa[4];
        sa[0] = Bf16::pack(S[2 * kk][0], S[2 * kk][1]);
        sa[1] = Bf16::pack(S[2 * kk][2], S[2 * kk][3]);
        sa[2] = Bf16::pack(S[2 * kk + 1][0], S[2 * kk + 1][1]);
        sa[3] = Bf16::pack(S[2 * kk + 1][2], S[2 * kk + 1][3]);
        float (&acc)[2][4] = cur ? u2 : u;
        mma16816<Bf16>(acc[0], sa, bw[cur][0], bw[cur][1]);
        mma16816<Bf16>(acc[1], sa, bw[cur][2], bw[cur][3]);
        mma16816<Bf16>(o[0], sa, bqd[cur][0], bqd[cur][1]);
        mma16816<Bf16>(o[1], sa, bqd[cur][2], bqd[cur][3]);
      }
      // the first k-step's operands of the state update
      const int k_row = (lane >> 4) * 8 + (lane & 7), k_half = (lane >> 3) & 1;
      uint32_t bk[2][4];
      float4 gq[2];
      ldsm_x4(bk[0], &sm.kr[0][0] + rt_cm_off(k_row, k_half));
      gq[0] = *reinterpret_cast<const float4*>(&sm.gamma[4 * t]);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) u[nt][e] += u2[nt][e];
      uint32_t ua[4];
      ua[0] = F16::pack(u[0][0], u[0][1]);
      ua[1] = F16::pack(u[0][2], u[0][3]);
      ua[2] = F16::pack(u[1][0], u[1][1]);
      ua[3] = F16::pack(u[1][2], u[1][3]);
      // S^T = S^T diag(gamma) + U^T k_res, operands one step ahead; gamma is indexed
      // by stored key: entries 0-1 are MMA keys 16 np + 2 t (+1), 2-3 are + 8
#pragma unroll
      for (int np = 0; np < KK; ++np) {
        const int cur = np & 1;
        if (np + 1 < KK) {
          ldsm_x4(bk[cur ^ 1], &sm.kr[0][0] + rt_cm_off(16 * (np + 1) + k_row, k_half));
          gq[cur ^ 1] = *reinterpret_cast<const float4*>(&sm.gamma[16 * (np + 1) + 4 * t]);
        }
        const float4 gm = gq[cur];
        S[2 * np][0] *= gm.x; S[2 * np][1] *= gm.y; S[2 * np][2] *= gm.x; S[2 * np][3] *= gm.y;
        mma16816<F16>(S[2 * np], ua, bk[cur][0], bk[cur][1]);
        S[2 * np + 1][0] *= gm.z; S[2 * np + 1][1] *= gm.w; S[2 * np + 1][2] *= gm.z; S[2 * np + 1][3] *= gm.w;
        mma16816<F16>(S[2 * np + 1], ua, bk[cur][2], bk[cur][3]);
      }
      // O^T += U^T Mqk^T
      {
        uint32_t bm[4];
        const int row = ((lane >> 4) << 3) + (lane & 7);
        ldsm_x4(bm, &sm.mqk[row][((lane >> 3) & 1) * 8]);
        mma16816<F16>(o[0], ua, bm[0], bm[1]);
        mma16816<F16>(o[1], ua, bm[2], bm[3]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int tok = 8 * nt + 2 * t;
        st.ostage[tok][r0 + g] = __float2bfloat16_rn(o[nt][0]);
        st.ostage[tok + 1][r0 + g] = __float2bfloat16_rn(o[nt][1]);
        st.ostage[tok][r0 + g + 8] = __float2bfloat16_rn(o[nt][2]);
        st.ostage[tok + 1][r0 + g + 8] = __float2bfloat16_rn(o[nt][3]);
      }
      // Between chunks the tile waits in tensor memory (each warp rereads only its
      // own tiles, after the next chunk's preparation) rather than in registers held
      // across the preparation; after the last chunk it goes back to its slot.
      if (kTmemState && c + 1 < nch) {
        if constexpr (kTmemState) tc05::st64_wait(taddr, s_cols);
      } else {  // (at d_k = 64 also between chunks: an L2 round trip)
#pragma unroll
        for (int pp = 0; pp < NT / 2; ++pp) {
          float4* d0 = reinterpret_cast<float4*>(S_slot + (r0 + g) * K + 16 * pp + 4 * t);
          float4* d1 = reinterpret_cast<float4*>(S_slot + (r0 + g + 8) * K + 16 * pp + 4 * t);
          const float4 x = make_float4(S[2 * pp][0], S[2 * pp][1], S[2 * pp + 1][0], S[2 * pp + 1][1]);
          const float4 y = make_float4(S[2 * pp][2], S[2 * pp][3], S[2 * pp + 1][2], S[2 * pp + 1][3]);
          if (c + 1 < nch) {
            __stcg(d0, x);
            __stcg(d1, y);
          } else {
            __stcs(d0, x);
            __stcs(d1, y);
          }
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < ntok * (V / 8); i += NTHR) {
      const int row = i / (V / 8), v8 = i - row * (V / 8);
      __nv_bfloat16* dst =
          reinterpret_cast<__nv_bfloat16*>(p.o) + ((static_cast<size_t>(b) * T + tok0 + row) * p.HV + hv) * V + v8 * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&st.ostage[row][v8 * 8]);
    }
    __syncthreads();  // the next chunk's preparation reuses every buffer above
  }
  if (resident) {  // every warp's tensor-memory accesses were waited for before this point
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      tc05::fence_after_sync();
      tc05::tmem_dealloc(sm.tmem_base, kTmemCols);
    }
  }
}

template <int K, int V, bool L2N, bool RES>
cudaError_t launch_rtc_t(const RecurrentCall& c, cudaStream_t s) {
  using Q = typename std::conditional_t<L2N, F16, Bf16>::T;
  constexpr size_t smem = sizeof(RtcSmem<K, V, Q>);
  static std::atomic<uint64_t> smem_set{0};
  {
    const cudaError_t e = set_smem_limit_once(kda_recurrent_tc_kernel<K, V, L2N, RES>, smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = static_cast<unsigned>(c.B) * static_cast<unsigned>(c.HV);
  kda_recurrent_tc_kernel<K, V, L2N, RES><<<grid, 128, smem, s>>>(c);
  return cudaGetLastError();
}

template <int K, int V, bool RES>
cudaError_t launch_rtc_kvr(const RecurrentCall& c, cudaStream_t s) {
  return c.l2norm ? launch_rtc_t<K, V, true, RES>(c, s) : launch_rtc_t<K, V, false, RES>(c, s);
}

template <int K, int V>
cudaError_t launch_rtc_kv(const RecurrentCall& c, cudaStream_t s) {
  if constexpr (K == 128) {
    if (c.T > 16) return launch_rtc_kvr<K, V, true>(c, s);
  }
  return launch_rtc_kvr<K, V, false>(c, s);
}

}  // namespace

cudaError_t launch_recurrent_tc(const RecurrentCall& c, cudaStream_t s) {
  if (c.B == 0) return cudaSuccess;
  if (c.T < 1 || c.T > kMaxT) return cudaErrorInvalidValue;
  if (c.K == 128 && c.V == 128) return launch_rtc_kv<128, 128>(c, s);
  if (c.K == 128 && c.V == 64) return launch_rtc_kv<128, 64>(c, s);
  if (c.K == 64 && c.V == 128) return launch_rtc_kv<64, 128>(c, s);
  if (c.K == 64 && c.V == 64) return launch_rtc_kv<64, 64>(c, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
