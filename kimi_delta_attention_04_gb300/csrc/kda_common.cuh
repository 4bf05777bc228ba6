// Device helpers shared by the KDA kernels: warp-level tensor-core MMA
// (mma.sync m16n8k16, fp32 accumulation), ldmatrix, cp.async, packing and
// warp reductions. sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kda_internal.h"

namespace kda {

// Raises `kernel`'s dynamic shared-memory limit to `bytes` once per device: the
// attribute belongs to each device's context, so a process driving several
// GPUs must set it on each. `done` is the kernel's record of the devices
// already set (ids 0-63; beyond that every call sets it).
template <typename Kernel>
inline cudaError_t set_smem_limit_once(Kernel kernel, size_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// ---------------------------------------------------------------------------
// Element types of MMA operands
// ---------------------------------------------------------------------------
struct Bf16 {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ T cvt(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float to_float(T x) { return __bfloat162float(x); }
};

struct F16 {
  using T = __half;
  // Saturating conversion: values beyond the fp16 range become +-65504, never inf.
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  static __device__ __forceinline__ T cvt(float x) {
    uint32_t r = pack(x, 0.f);
    return *reinterpret_cast<__half*>(&r);
  }
  static __device__ __forceinline__ float to_float(T x) { return __half2float(x); }
};

// D = A * B + D for one m16n8k16 tile; A 16x16 (row), B 16x8 (col), fp32 accumulators.
template <typename Op>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<Bf16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma16816<F16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Four 8x8 b16 matrices; lane l supplies the row address of matrix l/8, row l%8.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}

// 16-byte asynchronous global -> shared copy (L2-only caching).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Sum of 16 per-lane values over the warp. On return the total of value j sits
// in lanes 2j and 2j+1, i.e. lane l holds the total of value (l >> 1) & 15.
// 16 shuffles for 16 reductions (each round halves the values a lane keeps).
__device__ __forceinline__ float warp_transpose_reduce16(float (&v)[16], int lane) {
  float w8[8], w4[4], w2[2];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float send = up ? v[i] : v[i + 8];
      float keep = up ? v[i + 8] : v[i];
      w8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float send = up ? w8[i] : w8[i + 4];
      float keep = up ? w8[i + 4] : w8[i];
      w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float send = up ? w4[i] : w4[i + 2];
      float keep = up ? w4[i + 2] : w4[i];
      w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  float w1;
  {
    const bool up = lane & 2;
    float send = up ? w2[0] : w2[1];
    float keep = up ? w2[1] : w2[0];
    w1 = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return w1 + __shfl_xor_sync(0xffffffffu, w1, 1);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------------------
// 16x16 matrices held in registers in the mma.sync accumulator layout
// ---------------------------------------------------------------------------
// c[nt][e] = M[g + 8 (e >> 1)][8 nt + 2 t + (e & 1)], g = lane / 4, t = lane % 4.
struct Frag16 {
  float c[2][4];
};

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// A-operand fragments (m16 x k16) of M: the accumulator layout of two adjacent
// n-tiles is exactly the A layout.
template <typename Op>
__device__ __forceinline__ void frag_as_a(const Frag16& m, uint32_t (&a)[4]) {
  a[0] = Op::pack(m.c[0][0], m.c[0][1]);
  a[1] = Op::pack(m.c[0][2], m.c[0][3]);
  a[2] = Op::pack(m.c[1][0], m.c[1][1]);
  a[3] = Op::pack(m.c[1][2], m.c[1][3]);
}

// B-operand fragments (k16 x n8, k = row of M) for both n-tiles: each packed
// 8x8 block of the accumulator layout is transposed in registers.
template <typename Op>
__device__ __forceinline__ void frag_as_b(const Frag16& m, uint32_t (&b)[2][2]) {
  b[0][0] = movmatrix_trans(Op::pack(m.c[0][0], m.c[0][1]));  // rows 0-7,  cols 0-7
  b[0][1] = movmatrix_trans(Op::pack(m.c[0][2], m.c[0][3]));  // rows 8-15, cols 0-7
  b[1][0] = movmatrix_trans(Op::pack(m.c[1][0], m.c[1][1]));  // rows 0-7,  cols 8-15
  b[1][1] = movmatrix_trans(Op::pack(m.c[1][2], m.c[1][3]));  // rows 8-15, cols 8-15
}

template <typename Op>
__device__ __forceinline__ Frag16 frag_mm(const Frag16& A, const Frag16& B) {
  uint32_t a[4], b[2][2];
  frag_as_a<Op>(A, a);
  frag_as_b<Op>(B, b);
  Frag16 C;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    C.c[nt][0] = C.c[nt][1] = C.c[nt][2] = C.c[nt][3] = 0.f;
    mma16816<Op>(C.c[nt], a, b[nt][0], b[nt][1]);
  }
  return C;
}

__device__ __forceinline__ Frag16 frag_plus_identity(Frag16 m, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((e >> 1) == nt && g == 2 * t + (e & 1)) m.c[nt][e] += 1.f;
  return m;
}

// (I + L)^{-1} for a strictly lower-triangular 16x16 L, from X = -L in
// registers (accumulator layout): the Neumann series of X, which is exact
// because L^16 = 0, summed as (I + X)(I + X^2)(I + X^4)(I + X^8). Independent
// products are paired so the dependent chain is four products deep. One warp;
// operands rounded to Op.
template <typename Op>
__device__ __forceinline__ Frag16 neumann_inverse16_frag(const Frag16& X, int lane) {
  const Frag16 X2 = frag_mm<Op>(X, X);
  const Frag16 X4 = frag_mm<Op>(X2, X2);
  const Frag16 P1 = frag_mm<Op>(frag_plus_identity(X, lane), frag_plus_identity(X2, lane));
  const Frag16 X8 = frag_mm<Op>(X4, X4);
  const Frag16 P2 = frag_mm<Op>(P1, frag_plus_identity(X4, lane));
  return frag_mm<Op>(P2, frag_plus_identity(X8, lane));
}

// The same with L read from shared memory (row stride `ld` floats).
template <typename Op>
__device__ __forceinline__ Frag16 neumann_inverse16(const float* L, int ld, int lane) {
  const int g = lane >> 2, t = lane & 3;
  Frag16 X;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) X.c[nt][e] = -L[(g + 8 * (e >> 1)) * ld + 8 * nt + 2 * t + (e & 1)];
  return neumann_inverse16_frag<Op>(X, lane);
}

// 2^x and log2(x) straight from the special-function unit (PTX ex2.approx /
// lg2.approx: relative error about 2^-22; ftz: results below 2^-126 become 0).
// The decay factors need absolute accuracy near 1e-7 only, which these give in
// one instruction each.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus with the usual linear branch above 20 (the two differ by < 2.1e-9 there).
__device__ __forceinline__ float softplus_f(float x) { return x <= 20.f ? log1pf(expf(x)) : x; }

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// Chunk bookkeeping shared by the chunk kernels
// ---------------------------------------------------------------------------
constexpr int kChunk = 16;

// Position of one chunk: sequence n, chunk c within it, first global token and
// number of real tokens (1..16).
struct ChunkPos {
  int n, c, tok0, ntok;
};

// Maps a global chunk index to its sequence. Returns false past the last chunk
// or when the varlen plan was rejected.
__device__ __forceinline__ bool locate_chunk(const ChunkGeom& geo, int cg, ChunkPos& pos) {
  if (geo.cu_seqlens == nullptr) {
    const int n = cg / geo.chunks_per_seq;
    if (n >= geo.N) return false;
    const int c = cg - n * geo.chunks_per_seq;
    pos.n = n;
    pos.c = c;
    pos.tok0 = n * geo.T + c * kChunk;
    pos.ntok = min(kChunk, geo.T - c * kChunk);
    return pos.ntok > 0;
  }
  const int32_t* off = geo.chunk_off;
  if (off[geo.N + 1] != 1) return false;  // plan flag: cu_seqlens rejected
  if (cg >= off[geo.N]) return false;
  int lo = 0, hi = geo.N - 1;  // largest n with off[n] <= cg
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= cg) lo = mid; else hi = mid - 1;
  }
  pos.n = lo;
  pos.c = cg - off[lo];
  const int s = geo.cu_seqlens[lo], e = geo.cu_seqlens[lo + 1];
  pos.tok0 = s + pos.c * kChunk;
  pos.ntok = min(kChunk, e - pos.tok0);
  return pos.ntok > 0;
}

// Sequence bounds and first global chunk of sequence n. Returns false when the
// varlen plan was rejected.
__device__ __forceinline__ bool locate_seq(const ChunkGeom& geo, int n, int& tok_start, int& tok_end,
                                           int& chunk_base) {
  if (geo.cu_seqlens == nullptr) {
    tok_start = n * geo.T;
    tok_end = tok_start + geo.T;
    chunk_base = n * geo.chunks_per_seq;
    return true;
  }
  if (geo.chunk_off[geo.N + 1] != 1) return false;
  tok_start = geo.cu_seqlens[n];
  tok_end = geo.cu_seqlens[n + 1];
  chunk_base = geo.chunk_off[n];
  return true;
}

}  // namespace kda
