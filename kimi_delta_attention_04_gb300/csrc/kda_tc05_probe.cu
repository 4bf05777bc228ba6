// Diagnostic kernel for the 5th-generation tensor cores (tcgen05): one CTA
// computes D [128 x N] = A [128 x K] B^T (B given as [N x K]) with bf16 operands
// and fp32 accumulation in tensor memory, reads D back with tcgen05.ld and
// writes it to global memory, so a test can compare it with a host matmul (this
// pins the descriptor and layout encodings of kda_tcgen05.cuh). It then times
// `reps` single round trips (MMA issue -> commit seen on the mbarrier -> D in
// registers), one burst of `reps` back-to-back MMA groups on one accumulator
// and one burst that rotates over independent accumulators, in SM cycles.
//
// Every mbarrier wait is bounded (2 s); on expiry the kernel reports
// KDA_ERR_TIMEOUT, skips the remaining work and still frees its tensor memory.
#include "kda_cluster.cuh"
#include "kda_tcgen05.cuh"

namespace kda {
namespace {

constexpr int kPM = 128;
constexpr int kPMaxK = 128;
constexpr int kPMaxN = 256;
constexpr uint32_t kPCols = 512;   // whole TMEM of the SM: D in columns 0 .. N-1, A (if used) from kPACol
constexpr uint32_t kPACol = 256;   // K / 2 <= 64 columns of packed bf16 pairs
constexpr uint64_t kPWaitNs = 2000000000ull;

struct __align__(1024) ProbeSmem {
  unsigned char a[kPM * kPMaxK * 2];     // 32 KB, 1024-aligned (128-byte swizzle atoms)
  unsigned char b[kPMaxN * kPMaxK * 2];  // 64 KB
  uint64_t bar;
  uint32_t tmem_base;
};
constexpr size_t kProbeSmemBytes = sizeof(ProbeSmem) + 1024;  // + room to align the base to 1024

// Byte offset of element (row, k) of a K-major tile with `rows` rows and K
// columns (bf16): layout 0 = core matrices without swizzle, K / 8 of them per
// 8-row group; layout 1 = 128-byte swizzle, K split into 64-wide regions of
// rows x 128 bytes.
__device__ __forceinline__ uint32_t tile_off(int row, int k, int rows, int K, int layout) {
  if (layout == 0) return (row >> 3) * (K * 16) + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2;
  const int kk = k & 63;
  return (k >> 6) * (rows * 128) + row * 128 + ((((kk >> 3) ^ row) & 7) << 4) + (kk & 7) * 2;
}

// Descriptor of the [rows x 16] slice at K offset 16 s.
__device__ __forceinline__ uint64_t tile_desc(uint32_t base, int s, int rows, int K, int layout) {
  if (layout == 0) return tc05::smem_desc(base + s * 256, 128, K * 16, tc05::kSwizzleNone);
  const int k0 = 16 * s;
  return tc05::smem_desc(base + (k0 >> 6) * (rows * 128) + (k0 & 63) * 2, 16, 1024, tc05::kSwizzle128B);
}

__global__ void __launch_bounds__(128, 1)
    kda_tc05_probe_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, float* __restrict__ D,
                          int K, int N, int layout, int a_tmem, int reps, long long* cycles, int32_t* err) {
  extern __shared__ unsigned char probe_raw[];
  ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>((reinterpret_cast<uintptr_t>(probe_raw) + 1023) & ~uintptr_t{1023});
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) {
    tc05::tmem_alloc(&sm.tmem_base, kPCols);
    tc05::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // operands into shared memory, 16 bytes at a time
  for (int row = tid; row < kPM; row += 128)
    for (int k = 0; k < K; k += 8)
      *reinterpret_cast<uint4*>(sm.a + tile_off(row, k, kPM, K, layout)) =
          *reinterpret_cast<const uint4*>(A + static_cast<size_t>(row) * K + k);
  for (int row = tid; row < N; row += 128)
    for (int k = 0; k < K; k += 8)
      *reinterpret_cast<uint4*>(sm.b + tile_off(row, k, N, K, layout)) =
          *reinterpret_cast<const uint4*>(B + static_cast<size_t>(row) * K + k);
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tbase = sm.tmem_base;
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  if (a_tmem) {  // row tid of A as K / 2 packed pairs in columns kPACol ..
    for (int s = 0; s < K / 16; ++s) {
      uint32_t w[8];
      const uint4* src = reinterpret_cast<const uint4*>(A + static_cast<size_t>(tid) * K + 16 * s);
      const uint4 lo = src[0], hi = src[1];
      w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
      w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
      tc05::st8_wait(tbase + lane_base + kPACol + 8 * s, w);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc05::fence_before_sync();
  __syncthreads();

  const uint32_t idesc = tc05::idesc_f16kind(kPM, N, true);
  const uint32_t sa = smem_u32(sm.a), sb = smem_u32(sm.b);
  auto issue = [&] {
    for (int s = 0; s < K / 16; ++s) {
      const uint64_t bd = tile_desc(sb, s, N, K, layout);
      if (a_tmem)
        tc05::mma_ts(tbase, tbase + kPACol + 8 * s, bd, idesc, s > 0 ? 1u : 0u);
      else
        tc05::mma_ss(tbase, tile_desc(sa, s, kPM, K, layout), bd, idesc, s > 0 ? 1u : 0u);
    }
  };
  uint32_t phase = 0;
  bool failed = false;
  if (tid == 0) {
    tc05::fence_after_sync();
    issue();
    tc05::commit(&sm.bar);
  }
  if (!mbar_wait_bounded(smem_u32(&sm.bar), phase, kPWaitNs)) {
    failed = true;
    if (lane == 0) set_err(err, 4 /* KDA_ERR_TIMEOUT */);
  }
  phase ^= 1u;
  tc05::fence_after_sync();
  if (!__any_sync(0xffffffffu, failed)) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t r[16];
      tc05::ld16_wait(tbase + lane_base + c0, r);
      float* dst = D + static_cast<size_t>(tid) * N + c0;
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[j] = __uint_as_float(r[j]);
    }
  }
  failed = __syncthreads_or(failed);

  // round trips: issue -> completion seen -> D in registers (warp 0 waits and loads)
  long long t_done = 0, t_data = 0, t_burst = 0;
  for (int rep = 0; rep < reps && !failed; ++rep) {
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      long long t0 = 0;
      if (lane == 0) {
        tc05::fence_after_sync();
        t0 = clock64();
        issue();
        tc05::commit(&sm.bar);
      }
      bool ok = mbar_wait_bounded(smem_u32(&sm.bar), phase, kPWaitNs);
      const long long t1 = clock64();
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc05::fence_after_sync();
        uint32_t r[16];
        tc05::ld16_wait(tbase, r);
        const long long t2 = clock64();
        if (lane == 0) {
          t_done += t1 - t0;
          t_data += t2 - t0;
        }
      } else {
        failed = true;
        if (lane == 0) set_err(err, 4);
      }
    }
    phase ^= 1u;
    failed = __syncthreads_or(failed);
  }
  // burst: `reps` MMA groups back to back, one commit; also the cycles until the
  // last MMA has been issued (the issuing thread's own cost)
  long long t_issue = 0;
  if (reps > 0 && !failed) {
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      long long t0 = 0;
      if (lane == 0) {
        tc05::fence_after_sync();
        t0 = clock64();
        for (int rep = 0; rep < reps; ++rep) issue();
        t_issue = clock64() - t0;
        tc05::commit(&sm.bar);
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&sm.bar), phase, kPWaitNs));
      if (lane == 0) {
        if (ok) t_burst = clock64() - t0;
        else set_err(err, 4);
      }
    }
    phase ^= 1u;
  }
  // burst with independent accumulators: group j writes columns (j % nt) N ..,
  // so consecutive groups do not depend on each other
  long long t_indep = 0;
  const int nt = min(8, static_cast<int>((a_tmem ? kPACol : kPCols) / N));
  if (reps > 0 && !failed && nt > 1) {
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      long long t0 = 0;
      if (lane == 0) {
        tc05::fence_after_sync();
        t0 = clock64();
        for (int rep = 0; rep < reps; ++rep) {
          const uint32_t dcol = static_cast<uint32_t>((rep % nt) * N);
          for (int s = 0; s < K / 16; ++s) {
            const uint64_t bd = tile_desc(sb, s, N, K, layout);
            if (a_tmem)
              tc05::mma_ts(tbase + dcol, tbase + kPACol + 8 * s, bd, idesc, s > 0 ? 1u : 0u);
            else
              tc05::mma_ss(tbase + dcol, tile_desc(sa, s, kPM, K, layout), bd, idesc, s > 0 ? 1u : 0u);
          }
        }
        tc05::commit(&sm.bar);
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&sm.bar), phase, kPWaitNs));
      if (lane == 0) {
        if (ok) t_indep = clock64() - t0;
        else set_err(err, 4);
      }
    }
    phase ^= 1u;
  }
  if (tid == 0 && cycles != nullptr) {
    cycles[0] = t_done;
    cycles[1] = t_data;
    cycles[2] = t_burst;
    cycles[3] = reps;
    cycles[4] = t_indep;
    cycles[5] = nt > 1 ? nt : 0;
    cycles[6] = t_issue;
  }
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tbase, kPCols);
  }
}

}  // namespace

cudaError_t launch_tc05_probe(const void* a, const void* b, float* d, int K, int N, int layout, int a_tmem, int reps,
                              long long* cycles, int32_t* err, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_limit_once(kda_tc05_probe_kernel, kProbeSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  kda_tc05_probe_kernel<<<1, 128, kProbeSmemBytes, s>>>(static_cast<const uint16_t*>(a),
                                                        static_cast<const uint16_t*>(b), d, K, N, layout, a_tmem,
                                                        reps, cycles, err);
  return cudaGetLastError();
}

}  // namespace kda
