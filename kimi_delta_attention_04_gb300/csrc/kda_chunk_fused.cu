// Fused chunkwise KDA forward for bf16 inputs, dk = dv = 128: one 4-CTA
// thread-block cluster per (sequence, head), prep and recurrence in one kernel.
//
// Mathematics as in kda_chunk_tc.cu ("FlashKDA里的L矩阵和Mqk矩阵": L, Mqk, the
// Neumann inverse, the K2 chunk step; the sequence kept out of the grid and d_v
// split across CTAs as in "TileLang 实战：KDA 从零到一" §6.4). What changes is the
// placement:
//
//  * CTA r of the cluster owns value rows [32r, 32r + 32) of the state. Each of
//    its two recurrence warps owns 16 of those rows and all 128 keys: S^T
//    [16 x 128] fp32 in registers as sixteen m16n8 mma.sync accumulators, so
//    every contraction over the keys stays inside the warp (no exchange
//    between warps on the serial path), and two n-tiles of an accumulator are
//    one A fragment, so S^T and U^T enter their next MMAs by a conversion
//    alone. q_dec^T and k_res are B operands loaded from the channel-major
//    tiles; -W'^T and U~'^T arrive in the warp's register order. O^T (S^T
//    q_dec^T + U^T Mqk^T) is staged in shared memory; an output warp stores o,
//    off the serial path. The recurrence warps issue from SM sub-partitions 0
//    and 1 and the prep warps from 2 and 3, so the chain never shares a
//    scheduler with the prep.
//  * The same CTA's prep warps prepare every 4th chunk (chunks c = r mod 4):
//    gate, beta, L2 norm, decay products, L / Mqk, Neumann inverse, W and U~.
//    Two groups of four warps take alternate ones, each loading its next
//    chunk's input tiles with TMA as soon as the current ones are in registers.
//  * Prepared chunks travel through a ring of kGRing slots in global memory
//    (L2-resident; one ring per cluster, taken from a pool in the workspace):
//    the prep warps write the chunk straight into slot c mod kGRing (mostly
//    16-byte stores of channel-major tiles); the publisher warp then makes it
//    visible at cluster scope (fence.acq_rel.cluster) and arrives on the
//    slot's "ready" mbarrier in all four CTAs. Each CTA's mover warp bulk-loads the shared operands and its
//    own 32 rows of U~ into local stage c mod kRing and, when its recurrence
//    warps release that stage, hands the global slot back to the producer
//    ("gfree"). On GB300 an L2 bulk load delivers ~50 B/clk per SM against
//    ~15-25 B/clk for a push over distributed shared memory.
//  * Every mbarrier wait is bounded (KDA_ERR_TIMEOUT in err on expiry); loop trip
//    counts never depend on a wait, so named barriers stay matched and every CTA
//    reaches the closing cluster barrier.
#include <type_traits>

#include "kda_cluster.cuh"
#include "kda_common.cuh"
#include "kda_tma.h"

namespace kda {
namespace {

constexpr int FD = 128;              // dk = dv
constexpr int kCtas = 4;             // cluster size
constexpr int kRows = FD / kCtas;    // value rows per CTA
constexpr int kRing = 4;             // local stages per CTA
constexpr int kGRing = 16;           // global ring slots per cluster (a multiple of kCtas)
constexpr int kPool = 40;            // cluster rings in the workspace pool (> clusters resident at once)
constexpr int kRecWarps = 2;         // recurrence warps, 16 value rows each
// 16 warps. A warp issues from sub-partition (warp id mod 4); the serial
// recurrence gets sub-partitions 0 and 1 to itself and the light roles, the
// eight prep warps take sub-partitions 2 and 3:
//   warps 0, 1: recurrence; 4: mover; 5: publisher; 13: output; 8, 9, 12: idle
//   (the output pass, which has no chain, runs warps 8, 9 as a second
//   recurrence pair on the odd chunks); warps 2, 3, 6, 7: prep group 0;
//   10, 11, 14, 15: prep group 1.
constexpr int kFusedThreads = 512;
constexpr int kMoverWarp = 4, kPublisherWarp = 5, kOutputWarp = 13;
// Channel-major 16-bit tiles [channel][16 tokens]: one channel's 16 tokens are
// one 32-byte row, so the thread that owns a channel writes it with two 16-byte
// stores. The two 16-byte halves (tokens 0-7, 8-15) are swapped on rows whose
// bit 2 is set, so the eight rows one ldmatrix 8x8 load reads fall on distinct
// banks. cm_off gives the element offset of half `half` of row `row`.
__device__ __forceinline__ int cm_off(int row, int half) { return row * 16 + ((half ^ (row >> 2)) & 1) * 8; }
// Key order of the recurrence. It holds S^T [value x key] as m16n8 accumulators
// whose n-tile nt covers MMA keys 8 nt .. 8 nt + 7. Within each block of 16
// keys, the key the MMAs call 8 j + 2 t + e (n-tile j of the pair, column pair
// of lane t) is stored key 4 t + 2 j + e, so the four keys a lane holds over a
// pair of n-tiles are consecutive in memory and a state row moves as one
// 16-byte access per pair. The prep thread that writes row r of the
// key-indexed operand tiles (q_dec, k_res, k_dec and so -W) takes its q, k and
// gate from stored key key_of_mma_row(r); the level tiles sum over every key
// and do not care which.
__device__ __forceinline__ int key_of_mma_row(int r) {
  const int x = r & 15;
  return (r & ~15) + ((x >> 1) & 3) * 4 + ((x >> 3) & 1) * 2 + (x & 1);
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// -W'^T and U~'^T travel in the recurrence's register order. W[kk][lane] holds
// lane's B fragments of -W'^T for keys 16 kk .. 16 kk + 15 (token tiles 0 and 1);
// ut[m][j][lane] holds lane's accumulator of U~'^T for value rows 16 m .. 16 m +
// 15 and tokens 8 j .. 8 j + 7. The prep lane that computes them and the
// recurrence lane that uses them are the same (g, t), so each moves them as one
// 16-byte access. gamma is indexed by stored key: a lane's four decay factors
// of a pair of n-tiles are then one 16-byte load.
// The chunk operands are those of the unnormalised q, k (the L2 norm is folded
// in, see the prep): U' = diag(rk) U is the U operand, o_i = sr_i O'_i with
// O' = qd S + mqk U' and sr_i = scale rq_i.
struct __align__(16) Stage {
  uint4 W[FD / 16][32];    // bf16 pairs, -W'^T = -(diag(rk) INV diag(beta rk) k_dec)^T, B fragments
  uint16_t qd[FD][16];     // bf16, (q e^{G})^T, channel-major
  uint16_t kr[FD][16];     // st2, (k e^{G_last - G})^T, channel-major
  uint16_t mqk[16][24];    // st2, raw q_i . k_j e^{G_i - G_j} (j <= i)
  float gamma[FD];         // e^{G_last} by stored key
  float sr[16];            // output factor of each token: scale rq_i
  float4 ut[kRows / 16][2][32];  // U~'^T of this CTA's value rows, accumulators
};
constexpr uint32_t kSharedBytes = offsetof(Stage, ut);
constexpr uint32_t kUtSliceBytes = sizeof(float) * kRows * 16;
constexpr uint32_t kStageTx = kSharedBytes + kUtSliceBytes;
static_assert(kSharedBytes % 16 == 0 && kStageTx == sizeof(Stage), "stage layout");

struct __align__(16) PrepOut {
  uint4 W[FD / 16][32];
  uint16_t qd[FD][16];
  uint16_t kr[FD][16];
  uint16_t mqk[16][24];
  float gamma[FD];
  float sr[16];
  float4 ut[FD / 16][2][32];  // all value rows
};
static_assert(offsetof(PrepOut, ut) == kSharedBytes, "prep-out and stage share the layout");

constexpr uint32_t kSlotBytes = sizeof(PrepOut);
static_assert(kSlotBytes % 16 == 0, "slot size");
constexpr size_t kPoolHeader = 256;  // bitmap of the pool's rings in use
constexpr size_t kRingBytes = static_cast<size_t>(kGRing) * kSlotBytes;
static_assert(kPool <= 64, "bitmap holds 64 rings");

struct __align__(16) PrepIn {
  __nv_bfloat16 q[16][FD];
  __nv_bfloat16 k[16][FD];
  __nv_bfloat16 v[16][FD];
  float a[16][FD];  // gate inputs a, or log-decay g
};

template <typename Q>
struct __align__(16) PrepScratch {
  Q A_lv[4][FD][16];          // per level: [channel][row], channel-major
  Q B_lv[4][FD][8];           // per level: [channel][column]
  Q kdec[FD][16];             // channel-major
  __nv_bfloat16 vs[FD][16];   // channel-major
  float Lm[16][17];
  float Mq[16][17];
  float red[4][48];     // per warp: partial sums of q.q, k.k and q.k of the 16 tokens
  float beta[2][16];    // beta of the group's current / next chunk
  float ghead[2][16];   // per-head log-decay (KDA_GATE_HEAD_G) of the current / next chunk
  uint4 inv[32][3];  // INV' = (I + L)^{-1} diag(beta) from warp 0: per lane its A fragments (operand type, bf16 hi, lo)
};

constexpr int kOPitch = kRows + 4;  // padded row of the staged output (conflict-free reads)

struct __align__(16) RecScratch {
  float opart[kRing][16][kOPitch];  // [stage][token][value row]: O of the stage's chunk
};

// Output pass: each of the four recurrence warps (two pairs, even and odd
// chunks) keeps its 16 rows of the state entering its next chunk in s[wi][pair],
// bulk-loaded row by row (rows padded to 144 floats, so a quarter warp's
// 16-byte reads of rows g and g + 1 fall on distinct banks).
constexpr int kSnapPitch = FD + 16;
template <bool ON>
struct __align__(16) SnapStage {  // 16-byte rows: bulk-copy destinations and float4 reads
  float s[kRecWarps][2][16][kSnapPitch];
  uint64_t bar[kRecWarps][2];
};
template <>
struct SnapStage<false> {};

template <typename Q, int MODE>
struct __align__(128) FusedSmem {
  Stage ring[kRing];
  PrepIn pin[2];                   // input tiles of prep group g
  PrepScratch<Q> ps[2];            // scratch of prep group g
  RecScratch rs;
  uint64_t full[kRing];            // stage loaded (mover's bulk loads -> recurrence)
  uint64_t empty[kRing];           // stage released by the 4 recurrence warps and the output warp (-> mover)
  uint64_t ofull[kRing];           // O partials of the stage's chunk written (recurrence -> output warp)
  uint64_t ready[kGRing];          // global slot written and published (producer's publisher -> every mover)
  uint64_t gfree[kGRing];          // global slot read by all 4 CTAs (movers -> producer's prep)
  uint64_t sig[kGRing / kCtas];    // this CTA's slot written (prep -> publisher)
  uint64_t pinbar[2];              // input tiles of group g loaded (TMA -> prep)
  int ring_id;                     // pool ring of this cluster (CTA 0's copy is authoritative)
  SnapStage<MODE == 2> snap;
};

// Token of row r (column r) of a level's 8-row block, the level's half-block size
// being s = 2^ls (shifts: the level is a warp index, so a division would be a
// run-time one).
__device__ __forceinline__ int row_tok_f(int ls, int r) { return ((r >> ls) << (ls + 1)) + (1 << ls) + (r & ((1 << ls) - 1)); }
__device__ __forceinline__ int col_tok_f(int ls, int r) { return ((r >> ls) << (ls + 1)) + (r & ((1 << ls) - 1)); }

// One thread issues the TMA loads of one chunk's input tiles (16 tokens x 128
// channels of q, k, v and, with a gate, a or g) into a PrepIn buffer; the bytes
// are counted on that buffer's mbarrier. Tokens past the end read as zero;
// tokens of the next sequence are masked by the reader.
__device__ __forceinline__ void issue_inputs(const TmaInputMaps& m, PrepIn& in, uint64_t* bar, int h, int tok0,
                                             int gate_mode) {
  const bool gate_tile = gate_mode == 1 || gate_mode == 2;  // per-channel gate (not the per-head one)
  const uint32_t bytes = 3 * sizeof(in.q) + (gate_tile ? sizeof(in.a) : 0);
  mbar_arrive_expect_tx_local(bar, bytes);
  tma_load_3d(&in.q[0][0], &m.q, 0, h, tok0, bar);
  tma_load_3d(&in.k[0][0], &m.k, 0, h, tok0, bar);
  tma_load_3d(&in.v[0][0], &m.v, 0, h, tok0, bar);
  if (gate_tile) tma_load_3d(&in.a[0][0], &m.a, 0, h, tok0, bar);
}

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

// Takes a free ring of the workspace pool (a 64-bit map, cleared before the
// launch). The launcher has checked that at most kPool clusters of this kernel
// can be resident at once (~38 on GB300), so a ring is free whenever a cluster
// starts; the wait is bounded all the same. Returns -1 (and reports a timeout)
// on failure.
__device__ int claim_ring(unsigned char* pool, int32_t* err) {
  unsigned int* bits = reinterpret_cast<unsigned int*>(pool);
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int w = 0; w < 2; ++w) {
      const unsigned int valid = (w == 0) ? 0xffffffffu : ((1u << (kPool - 32)) - 1u);
      unsigned int free_bits = ~atomicOr(&bits[w], 0u) & valid;
      while (free_bits != 0u) {
        const int b = __ffs(free_bits) - 1;
        const unsigned int old = atomicOr(&bits[w], 1u << b);
        if ((old & (1u << b)) == 0u) return 32 * w + b;
        free_bits = ~old & valid;
      }
    }
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      set_err(err, 4 /* KDA_ERR_TIMEOUT */);
      return -1;
    }
    __nanosleep(1000);
  }
}

// MODE 0: the forward; 1: the forward writing the state entering every chunk
// to h_chunks; 2: the chunk-parallel output pass from those states.
template <bool DELTA, bool L2N, int MODE>
__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kFusedThreads, 1)
    kda_chunk_fused_kernel(const ChunkCall p, const __grid_constant__ TmaInputMaps maps) {
  using QK = std::conditional_t<L2N, F16, Bf16>;
  using ST2 = std::conditional_t<DELTA, F16, Bf16>;
  using Q = typename QK::T;
  using Smem = FusedSmem<Q, MODE>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

  const int H = p.geo.H;
  const uint32_t rank = cluster_ctarank();
  const int unit = blockIdx.x / kCtas;
  const int n = unit / H;
  const int h = unit - n * H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int ts = 0, te = 0, cb = 0;
  const bool located = locate_seq(p.geo, n, ts, te, cb);
  const int nch0 = located ? (te - ts + kChunk - 1) / kChunk : 0;

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kRecWarps + 1);
      mbar_init(&sm.ofull[s], kRecWarps);
    }
    for (int i = 0; i < kGRing; ++i) {
      mbar_init(&sm.ready[i], 1);
      mbar_init(&sm.gfree[i], kCtas);
    }
    for (int i = 0; i < kGRing / kCtas; ++i) mbar_init(&sm.sig[i], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.pinbar[b], 1);
    }
    if constexpr (MODE == 2)
      for (int w = 0; w < kRecWarps; ++w)
        for (int b = 0; b < 2; ++b) mbar_init(&sm.snap.bar[w][b], 1);
    sm.ring_id = (rank == 0 && nch0 > 0) ? claim_ring(p.records, p.err) : -1;
    fence_mbarrier_init_cluster();
  }
  cluster_sync_all();
  // every CTA works on CTA 0's ring; without one (nothing to do, or no ring
  // could be had) the cluster does nothing
  const int ring_id = ld_shared_cluster_s32(mapa_shared(smem_u32(&sm.ring_id), 0));
  const bool ok = located && (nch0 == 0 || ring_id >= 0);
  const int nch = ring_id >= 0 ? nch0 : 0;
  unsigned char* const gring =
      p.records + kPoolHeader + static_cast<size_t>(ring_id >= 0 ? ring_id : 0) * kRingBytes;

  if (warp < kRecWarps || (MODE == 2 && (warp == 8 || warp == 9))) {
    // ===================== recurrence warps =====================
    // Warp w owns value rows [dv0, dv0 + 16) of the CTA's 32 and all 128 keys:
    // S^T [16 x d_k] fp32 in registers as sixteen m16n8 accumulators, ST[nt] =
    // MMA keys 8 nt .. 8 nt + 7. Every contraction over d_k stays inside the
    // warp, and two n-tiles of an accumulator are one A fragment, so S^T and U^T
    // enter their next MMAs by a conversion alone:
    //   U^T = U~^T + S^T (-W)^T,  O^T = S^T q_dec^T + U^T Mqk^T,
    //   S^T <- S^T diag(gamma) + U^T k_res.
    const int g = lane >> 2, t = lane & 3;
    const int wi = warp & 1;                                 // which 16 of the CTA's value rows
    const int dvl = wi * 16;                                 // first value row within the CTA
    const int dv0 = static_cast<int>(rank) * kRows + dvl;   // first value row of the stored state
    // ldmatrix lane addresses (lane matrix m = lane / 8). B fragments of q_dec^T
    // ([key][token]) from .trans loads of the channel-major tile, m = (key half
    // m & 1, token half m >> 1); of k_res ([token][key]) from plain loads, m =
    // (key half m >> 1, token half m & 1); of Mqk^T from plain loads of the
    // row-major [i][j] tile, m = (i half m >> 1, j half m & 1).
    const int bq_row = ((lane >> 3) & 1) * 8 + (lane & 7), bq_half = lane >> 4;
    const int bk_row = (lane >> 4) * 8 + (lane & 7), bk_half = (lane >> 3) & 1;
    const int mq_row = (lane >> 4) * 8 + (lane & 7), mq_col = ((lane >> 3) & 1) * 8;
    // Output pass: no recurrence; each chunk's entering state comes from
    // h_chunks through the warp's snapshot buffer, and pair `pair` takes the
    // chunks of its parity.
    constexpr bool outp = MODE == 2;
    const int pair = outp ? (warp >> 3) : 0;
    constexpr int kStep = outp ? 2 : 1;
    float ST[16][4];
    // rows dv0 + g and dv0 + g + 8 of a stored [dv][dk] state: stored keys
    // 16 pp + 4 t .. + 3 are MMA keys 16 pp + 2 t (+1) and 16 pp + 8 + 2 t (+1)
    auto load_state = [&](const float* src) {
      const float* r0 = src + static_cast<size_t>(dv0 + g) * FD + 4 * t;
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(r0 + 16 * pp));
        const float4 y = __ldcs(reinterpret_cast<const float4*>(r0 + 8 * FD + 16 * pp));
        ST[2 * pp][0] = x.x; ST[2 * pp][1] = x.y; ST[2 * pp + 1][0] = x.z; ST[2 * pp + 1][1] = x.w;
        ST[2 * pp][2] = y.x; ST[2 * pp][3] = y.y; ST[2 * pp + 1][2] = y.z; ST[2 * pp + 1][3] = y.w;
      }
    };
    auto store_state = [&](float* dst, bool streaming) {
      float* r0 = dst + static_cast<size_t>(dv0 + g) * FD + 4 * t;
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        float4* d0 = reinterpret_cast<float4*>(r0 + 16 * pp);
        float4* d1 = reinterpret_cast<float4*>(r0 + 8 * FD + 16 * pp);
        const float4 x = make_float4(ST[2 * pp][0], ST[2 * pp][1], ST[2 * pp + 1][0], ST[2 * pp + 1][1]);
        const float4 y = make_float4(ST[2 * pp][2], ST[2 * pp][3], ST[2 * pp + 1][2], ST[2 * pp + 1][3]);
        if (streaming) {
          __stcs(d0, x);
          __stcs(d1, y);
        } else {
          *d0 = x;
          *d1 = y;
        }
      }
    };
    auto snapshot = [&](int cc) { return p.h_chunks + (static_cast<size_t>(cb + cc) * H + h) * FD * FD; };
    if (!outp) {
      if (ok && p.h0 != nullptr) {
        load_state(p.h0 + (static_cast<size_t>(n) * H + h) * FD * FD);
      } else {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) ST[nt][0] = ST[nt][1] = ST[nt][2] = ST[nt][3] = 0.f;
      }
    }
    bool failed = false;
    float o[2][4];  // O^T of the chunk: value rows g, g + 8, tokens 8 j + 2 t (+1)
    auto post_output = [&](int cc) {
      float (*op)[kOPitch] = sm.rs.opart[cc & (kRing - 1)];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tk = 8 * j + 2 * t;
        op[tk][dvl + g] = o[j][0];
        op[tk + 1][dvl + g] = o[j][1];
        op[tk][dvl + g + 8] = o[j][2];
        op[tk + 1][dvl + g + 8] = o[j][3];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_local(&sm.ofull[cc & (kRing - 1)]);
    };
    // this CTA's 32 value rows of chunk cc's state: one contiguous 16 KB slab, pulled
    // into L2 kSnapAhead chunks before its loads (by the first warp of the pair)
    constexpr int kSnapAhead = 4;
    auto prefetch_state = [&](int cc) {
      if (wi == 0 && lane == 0 && cc < nch) bulk_prefetch_l2(snapshot(cc) + rank * kRows * FD, kRows * FD * 4);
    };
    // the warp's 16 rows of chunk cc's entering state into its snapshot buffer;
    // after a failed wait no new copy is started (decided for the whole warp)
    int snap_issued[2] = {-1, -1}, snap_seen[2] = {-1, -1};
    auto load_snap = [&](int cc) {
      if constexpr (outp) {
        if (cc < nch && !__any_sync(0xffffffffu, failed)) {
          snap_issued[cc & 1] = cc;
          uint64_t* bar = &sm.snap.bar[wi][cc & 1];
          if (lane == 0) mbar_arrive_expect_tx_local(bar, 16 * FD * 4);
          __syncwarp();
          if (lane < 16)
            bulk_load_g2s(&sm.snap.s[wi][cc & 1][lane][0], snapshot(cc) + static_cast<size_t>(dv0 + lane) * FD,
                          FD * 4, bar);
        }
      }
    };
    if (outp) {
      for (int cc = pair + 2; cc < pair + 2 + kSnapAhead; cc += 2) prefetch_state(cc);
      load_snap(pair);
    }
    // set mid-chunk when every lane's non-blocking test saw the next chunk's stage
    // loaded: its blocking wait (whose latency sits on the serial path) is skipped.
    // Not in the snapshot forward, which spills with it.
    constexpr bool kPretest = MODE != 1;
    bool next_ready = false;
    for (int c = pair; c < nch; c += kStep) {
      const int s = c & (kRing - 1);
      const uint32_t par = static_cast<uint32_t>(c / kRing) & 1u;
      const bool stage_ready = next_ready;
      next_ready = false;
      // the state entering chunk c (before its decay) goes to h_chunks one key
      // pair per step of the U loop below, where the MMAs leave issue slots free
      float* const snap_row = MODE == 1 ? snapshot(c) + static_cast<size_t>(dv0 + g) * FD + 4 * t : nullptr;
      if (!failed && !stage_ready && !mbar_wait_bounded(smem_u32(&sm.full[s]), par, kWaitLimitNs)) {
        failed = true;
        if (lane == 0) set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
      }
      if constexpr (outp) {
        if (!failed && !mbar_wait_bounded(smem_u32(&sm.snap.bar[wi][c & 1]), static_cast<uint32_t>(c >> 1) & 1u,
                                          kWaitLimitNs)) {
          failed = true;
          if (lane == 0) set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
        }
        if (!failed) snap_seen[c & 1] = c;
      }
      const Stage& st = sm.ring[s];
      // U^T = U~^T + S^T (-W)^T (the serial path, two accumulator chains per
      // token tile) and O^T = S^T q_dec^T, one key step of S^T at a time. The
      // MMAs and ldmatrix loads keep their program order, so each key step's
      // shared-memory operands are loaded one step ahead of their MMAs.
      uint32_t bq[2][4];
      uint4 wv[2];
      ldsm_x4_trans(bq[0], &st.qd[0][0] + cm_off(bq_row, bq_half));
      if (DELTA) wv[0] = st.W[0][lane];
      float u[2][4], u2[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float4 x = st.ut[wi][j][lane];
        u[j][0] = x.x; u[j][1] = x.y; u[j][2] = x.z; u[j][3] = x.w;
        u2[j][0] = u2[j][1] = u2[j][2] = u2[j][3] = 0.f;
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int cur = kk & 1;
        if (kk + 1 < 8) {
          ldsm_x4_trans(bq[cur ^ 1], &st.qd[0][0] + cm_off(16 * (kk + 1) + bq_row, bq_half));
          if (DELTA) wv[cur ^ 1] = st.W[kk + 1][lane];
        }
        uint32_t sa[4];
        if constexpr (outp) {
          const float* r0 = &sm.snap.s[wi][c & 1][g][16 * kk + 4 * t];
          const float4 x = *reinterpret_cast<const float4*>(r0);
          const float4 y = *reinterpret_cast<const float4*>(r0 + 8 * kSnapPitch);
          sa[0] = Bf16::pack(x.x, x.y);
          sa[1] = Bf16::pack(y.x, y.y);
          sa[2] = Bf16::pack(x.z, x.w);
          sa[3] = Bf16::pack(y.z, y.w);
        } else {
          sa[0] = Bf16::pack(ST[2 * kk][0], ST[2 * kk][1]);
          sa[1] = Bf16::pack(ST[2 * kk][2], ST[2 * kk][3]);
          sa[2] = Bf16::pack(ST[2 * kk + 1][0], ST[2 * kk + 1][1]);
          sa[3] = Bf16::pack(ST[2 * kk + 1][2], ST[2 * kk + 1][3]);
          if (MODE == 1) {
            __stcs(reinterpret_cast<float4*>(snap_row + 16 * kk),
                   make_float4(ST[2 * kk][0], ST[2 * kk][1], ST[2 * kk + 1][0], ST[2 * kk + 1][1]));
            __stcs(reinterpret_cast<float4*>(snap_row + 8 * FD + 16 * kk),
                   make_float4(ST[2 * kk][2], ST[2 * kk][3], ST[2 * kk + 1][2], ST[2 * kk + 1][3]));
          }
        }
        if (DELTA) {
          // The plain forward keeps one accumulator chain: under the 128-register
          // cap its body then runs faster than with two (measured); the snapshot
          // modes, which hold more registers, keep two.
          float (&acc)[2][4] = (cur && MODE != 0) ? u2 : u;
          mma16816<Bf16>(acc[0], sa, wv[cur].x, wv[cur].y);
          mma16816<Bf16>(acc[1], sa, wv[cur].z, wv[cur].w);
        }
        mma16816<Bf16>(o[0], sa, bq[cur][0], bq[cur][1]);
        mma16816<Bf16>(o[1], sa, bq[cur][2], bq[cur][3]);
      }
      if constexpr (kPretest) {  // the next chunk's stage, tested without blocking
        const int cn = c + kStep;
        const bool t_ok = cn < nch && mbar_test_wait(smem_u32(&sm.full[cn & (kRing - 1)]),
                                                     static_cast<uint32_t>(cn / kRing) & 1u);
        next_ready = __all_sync(0xffffffffu, t_ok);
      }
      // the operands of Mqk^T and of the first key step of the state update
      uint32_t bm[4], bk[2][4];
      float4 gq[2];
      ldsm_x4(bm, &st.mqk[mq_row][mq_col]);
      if (!outp) {
        ldsm_x4(bk[0], &st.kr[0][0] + cm_off(bk_row, bk_half));
        gq[0] = *reinterpret_cast<const float4*>(&st.gamma[4 * t]);
      }
      if constexpr (outp) {  // the snapshot buffer is read: refill it with the pair's next chunk
        __syncwarp();
        fence_proxy_async_smem();
        load_snap(c + 2);
        prefetch_state(c + 2 + kSnapAhead);
      }
      if (DELTA) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) u[j][e] += u2[j][e];
      }
      // U^T as an A fragment [value][token]
      uint32_t ua[4];
      ua[0] = ST2::pack(u[0][0], u[0][1]);
      ua[1] = ST2::pack(u[0][2], u[0][3]);
      ua[2] = ST2::pack(u[1][0], u[1][1]);
      ua[3] = ST2::pack(u[1][2], u[1][3]);
      if (!outp) {
        // S^T = S^T diag(gamma) + U^T k_res, keys 16 np .. 16 np + 15 at a time,
        // operands one step ahead
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          const int cur = np & 1;
          if (np + 1 < 8) {
            ldsm_x4(bk[cur ^ 1], &st.kr[0][0] + cm_off(16 * (np + 1) + bk_row, bk_half));
            gq[cur ^ 1] = *reinterpret_cast<const float4*>(&st.gamma[16 * (np + 1) + 4 * t]);
          }
          // decay of MMA keys 16 np + 2 t (+1) and 16 np + 8 + 2 t (+1)
          const float4 gm = gq[cur];
          ST[2 * np][0] *= gm.x; ST[2 * np][1] *= gm.y; ST[2 * np][2] *= gm.x; ST[2 * np][3] *= gm.y;
          ST[2 * np + 1][0] *= gm.z; ST[2 * np + 1][1] *= gm.w; ST[2 * np + 1][2] *= gm.z; ST[2 * np + 1][3] *= gm.w;
          mma16816<ST2>(ST[2 * np], ua, bk[cur][0], bk[cur][1]);
          mma16816<ST2>(ST[2 * np + 1], ua, bk[cur][2], bk[cur][3]);
          if (np == 0) {  // O^T += U^T Mqk^T, off the serial path
            mma16816<ST2>(o[0], ua, bm[0], bm[1]);
            mma16816<ST2>(o[1], ua, bm[2], bm[3]);
          }
        }
      } else {  // O^T += U^T Mqk^T
        mma16816<ST2>(o[0], ua, bm[0], bm[1]);
        mma16816<ST2>(o[1], ua, bm[2], bm[3]);
      }
      if constexpr (MODE == 0) {
        // the stage is read: released before the O stores, which go to another
        // buffer (measured faster in the forward; the snapshot modes spill with it)
        __syncwarp();
        if (lane == 0) mbar_arrive_local(&sm.empty[s]);
        post_output(c);
      } else {
        post_output(c);
        if (lane == 0) mbar_arrive_local(&sm.empty[s]);
      }
    }
    if (ok && p.hT != nullptr && !outp) store_state(p.hT + (static_cast<size_t>(n) * H + h) * FD * FD, false);
    if constexpr (outp) {  // no snapshot copy may still be landing when the CTA exits
#pragma unroll
      for (int b = 0; b < 2; ++b)
        if (snap_issued[b] > snap_seen[b] &&
            !mbar_wait_bounded(smem_u32(&sm.snap.bar[wi][b]), static_cast<uint32_t>(snap_issued[b] >> 1) & 1u,
                               kWaitLimitNs) &&
            lane == 0)
          set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
    }
  } else if ((warp & 3) >= 2) {
    // ===================== prep warps =====================
    // Chunk c is prepared in shared memory (pout), then copied into global slot
    // c mod kGRing once all four CTAs have loaded that slot's previous chunk.
    // Two groups of four warps; group g prepares this CTA's chunks j = g mod 2
    // (c = rank + 4 j), so two chunks are in flight and each group's latency
    // hides behind the other's.
    const int grp = warp >> 3;
    const int pt = 32 * (((warp >> 2) & 1) * 2 + (warp & 1)) + lane;  // value channel and key-operand row owned
    const int kc = key_of_mma_row(pt);     // the key channel behind that row
    const int pw = pt >> 5;                // warp index 0..3 within the group
    const uint32_t bar_id = grp == 0 ? 1u : 4u;
    auto prep_bar = [bar_id] { named_bar_sync(bar_id, 128); };
    PrepScratch<Q>& ps = sm.ps[grp];
    constexpr float kLog2e = 1.4426950408889634f;
    const float Aexp = (p.gate_mode == 2) ? expf(p.A_log[h]) : 0.f;
    const float dtb2 = (p.gate_mode == 2) ? p.dt_bias[h * FD + kc] * kLog2e : 0.f;  // dt_bias in log2 units
    bool failed = false;
    int c = static_cast<int>(rank) + kCtas * grp;
    // beta and the per-head gate of the group's chunks: lanes 0-15 of the
    // group's warp 1 load the raw values one chunk of the group ahead and, while
    // warp 0 forms the current chunk's inverse, turn them into
    // ps.beta / ps.ghead [buffer of that chunk].
    const int bl = pt - 32;  // token handled by warp 1's lanes 0-15
    const bool bown = bl >= 0 && bl < 16;
    unsigned short beta_next = 0;
    float gh_next = 0.f;
    auto load_next = [&](int cc) {
      const int tk0 = ts + cc * kChunk;
      beta_next = 0;
      gh_next = 0.f;
      if (bown && tk0 + bl < te) {
        if (DELTA) beta_next = reinterpret_cast<const unsigned short*>(p.beta)[static_cast<size_t>(tk0 + bl) * H + h];
        if (p.gate_mode == 3) gh_next = p.g[static_cast<size_t>(tk0 + bl) * H + h];
      }
    };
    auto stage_next = [&](int bufi, int cc) {
      if (bown) {
        const float raw = __bfloat162float(__ushort_as_bfloat16(beta_next));
        const float bt = (p.beta_mode == 1) ? sigmoid_f(raw) : raw;
        ps.beta[bufi][bl] = (DELTA && ts + cc * kChunk + bl < te) ? bt : 0.f;
        ps.ghead[bufi][bl] = gh_next;
      }
    };
    // Each group loads its own input tiles with TMA: the first chunk's now,
    // chunk c + 8's as soon as chunk c's are in registers.
    if (pt == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.q) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.k) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.v) : "memory");
      if (p.gate_mode == 1 || p.gate_mode == 2) asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.a) : "memory");
      if (c < nch) issue_inputs(maps, sm.pin[grp], &sm.pinbar[grp], h, ts + c * kChunk, p.gate_mode);
    }
    // the first chunk's beta and gate, and clear L / Mqk scratch (ordered by the
    // loop's first barrier)
    if (c < nch) {
      load_next(c);
      stage_next(0, c);
    }
    if (c + 2 * kCtas < nch) load_next(c + 2 * kCtas);
    for (int i = pt; i < 16 * 17; i += 128) {
      (&ps.Lm[0][0])[i] = 0.f;
      (&ps.Mq[0][0])[i] = 0.f;
    }
    // The hand-off of a written chunk to the publisher (a release at CTA scope)
    // is made after the next chunk's first barrier: right after the slot
    // stores it would wait for their L2 acknowledgements.
    int sig_pending = -1;
    auto signal_written = [&] {
      if (pt == 0 && sig_pending >= 0) mbar_arrive_local(&sm.sig[sig_pending % (kGRing / kCtas)]);
      sig_pending = -1;
    };
    // The L2 norm is folded into the chunk's small matrices instead of scaling
    // q and k: everything below uses the raw q~, k~ of the tokens, with
    // rq_i = 1 / |q~_i|, rk_i = 1 / |k~_i| (1 without the norm). Then
    //   L = diag(beta rk) (k~ k~^T . decay) diag(rk)       (the L of unit q, k)
    //   U' = diag(rk) U = INV_U v - INV_W k~_dec S,  INV_U = diag(rk) INV diag(beta),
    //                                                INV_W = INV_U diag(rk)
    //   S <- gamma S + k~_res^T U',   o_i = scale rq_i (q~_dec S + Mqk~ U')_i,
    // where Mqk~ holds the raw q~_i . k~_j decay products: exactly the
    // recurrence of unit q, k, with no pass over the 16 x 128 tiles for the norm
    // and no barrier waiting for it.
    for (int j = grp; c < nch; j += 2, c += 2 * kCtas) {
      const int buf = grp;
      const int jb = (j >> 1) & 1;  // beta / gate buffer of this chunk
      const int tok0 = ts + c * kChunk;
      const int ntok = min(kChunk, te - tok0);
      if (!failed && !mbar_wait_bounded(static_cast<uint32_t>(__cvta_generic_to_shared(&sm.pinbar[buf])),
                                        static_cast<uint32_t>(j >> 1) & 1u, kWaitLimitNs)) {
        failed = true;
        if (pt == 0) {
          set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
          // the copy waited for is the only one that can be in flight (none is
          // started after a failed wait): it gets one more bounded wait, so no
          // input copy lands once the CTA has exited
          mbar_wait_bounded(static_cast<uint32_t>(__cvta_generic_to_shared(&sm.pinbar[buf])),
                            static_cast<uint32_t>(j >> 1) & 1u, kWaitLimitNs);
        }
      }
      // the chunk is written straight into global slot c mod kGRing, once all
      // four CTAs have loaded that slot's previous chunk
      const int gs = c % kGRing;
      if (c >= kGRing && pt == 0 && !failed &&
          !mbar_wait_bounded(smem_u32(&sm.gfree[gs]), static_cast<uint32_t>(c / kGRing - 1) & 1u, kWaitLimitNs)) {
        failed = true;
        set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
      }
      PrepOut& po = *reinterpret_cast<PrepOut*>(gring + static_cast<size_t>(gs) * kSlotBytes);
      prep_bar();  // (A) this chunk's beta and gate staged, L / Mqk scratch clear
      signal_written();
      const PrepIn& in = sm.pin[buf];
      float qv[16], kv[16], al[16], vv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        qv[i] = __bfloat162float(in.q[i][kc]);
        kv[i] = __bfloat162float(in.k[i][kc]);
        vv[i] = __bfloat162float(in.v[i][pt]);
      }
      // One branch for the gate mode around the whole token loop, so the 16
      // independent exp/log chains interleave.
      if (p.gate_mode == 2) {
        // alpha = e^{-A softplus(x)} = 2^{-A log2(1 + 2^y)}, y = x log2 e. Above the
        // threshold x > 20 softplus(x) is x itself: log2(1 + 2^y) >= y always, and
        // with the exponent clamped at 20 log2 e the log stays below y there, so
        // max(log2(1 + 2^min(y, 20 log2 e)), y) is the thresholded softplus.
        constexpr float kClamp = 20.f * kLog2e;
        const float nA = -Aexp;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float y = fmaf(in.a[i][kc], kLog2e, dtb2);
          const float sp2 = fmaxf(lg2_approx(1.f + ex2_approx(fminf(y, kClamp))), y);
          al[i] = ex2_approx(nA * sp2);
        }
      } else if (p.gate_mode == 3) {
#pragma unroll
        for (int i = 0; i < 16; ++i) al[i] = ex2_approx(ps.ghead[jb][i] * kLog2e);
      } else if (p.gate_mode == 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) al[i] = ex2_approx(in.a[i][kc] * kLog2e);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) al[i] = 1.f;
      }
      if (ntok < 16) {  // the last chunk of a sequence (uniform across the CTA): rows past
                        // its end belong to another sequence or lie past the tensor
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i >= ntok) {
            qv[i] = kv[i] = vv[i] = 0.f;
            al[i] = 1.f;
          }
        }
      }
      {  // this warp's partial sums of q~.q~, k~.k~ and q~.k~ per token over its 32
         // channels: the diagonals of Q Q^T, K K^T and Q K^T on the tensor cores (bf16
         // products are exact in fp32). The warp stages raw channel-major rows of its
         // own 32 channels in level tiles 2 and 3, which the level operands below
         // overwrite; as A operands [token][channel] they come from .trans loads, and
         // the B fragments of Q^T (K^T) are the A fragments of Q (K) in another order.
        uint16_t* const rq_t = reinterpret_cast<uint16_t*>(&ps.A_lv[2][0][0]);
        uint16_t* const rk_t = reinterpret_cast<uint16_t*>(&ps.A_lv[3][0][0]);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = Bf16::pack(qv[2 * i], qv[2 * i + 1]);
        *reinterpret_cast<uint4*>(rq_t + cm_off(pt, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(rq_t + cm_off(pt, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = Bf16::pack(kv[2 * i], kv[2 * i + 1]);
        *reinterpret_cast<uint4*>(rk_t + cm_off(pt, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(rk_t + cm_off(pt, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        __syncwarp();
        // lane matrix m of an A fragment: (channel half m >> 1, token half m & 1)
        const int r_row = ((lane >> 4) & 1) * 8 + (lane & 7), r_half = (lane >> 3) & 1;
        float dqq[2][4] = {}, dkk[2][4] = {}, dqk[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t aq[4], ak[4];
          ldsm_x4_trans(aq, rq_t + cm_off(32 * pw + 16 * ks + r_row, r_half));
          ldsm_x4_trans(ak, rk_t + cm_off(32 * pw + 16 * ks + r_row, r_half));
          mma16816<Bf16>(dqq[0], aq, aq[0], aq[2]);
          mma16816<Bf16>(dqq[1], aq, aq[1], aq[3]);
          mma16816<Bf16>(dkk[0], ak, ak[0], ak[2]);
          mma16816<Bf16>(dkk[1], ak, ak[1], ak[3]);
          mma16816<Bf16>(dqk[0], aq, ak[0], ak[2]);
          mma16816<Bf16>(dqk[1], aq, ak[1], ak[3]);
        }
        // diagonal element (i, i): token tile i / 8, held by lane (g, g / 2) with
        // g = i % 8, entry (i % 8) % 2 (+2 in the second token tile)
        const int g = lane >> 2;
        if ((g >> 1) == (lane & 3)) {
          const int e = g & 1;
          ps.red[pw][g] = e ? dqq[0][1] : dqq[0][0];
          ps.red[pw][8 + g] = e ? dqq[1][3] : dqq[1][2];
          ps.red[pw][16 + g] = e ? dkk[0][1] : dkk[0][0];
          ps.red[pw][24 + g] = e ? dkk[1][3] : dkk[1][2];
          ps.red[pw][32 + g] = e ? dqk[0][1] : dqk[0][0];
          ps.red[pw][40 + g] = e ? dqk[1][3] : dqk[1][2];
        }
        __syncwarp();  // the staged rows are read before the level operands overwrite them
      }
      float P[16], Rs[16];
      P[0] = al[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) P[i] = P[i - 1] * al[i];
      Rs[15] = 1.f;
#pragma unroll
      for (int i = 14; i >= 0; --i) Rs[i] = Rs[i + 1] * al[i + 1];
      {
        // channel pt's 16 tokens of each channel-major tile, two 16-byte stores each,
        // at row `row` (the MMA key order for the key-indexed tiles, the channel
        // itself for the value and level tiles)
        auto put16 = [&](uint16_t* tile, const uint32_t (&w)[8], int row) {
          *reinterpret_cast<uint4*>(tile + cm_off(row, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(tile + cm_off(row, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        };
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = Bf16::pack(qv[2 * i] * P[2 * i], qv[2 * i + 1] * P[2 * i + 1]);
        put16(&po.qd[0][0], w, pt);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = ST2::pack(kv[2 * i] * Rs[2 * i], kv[2 * i + 1] * Rs[2 * i + 1]);
        put16(&po.kr[0][0], w, pt);
        if (DELTA) {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = QK::pack(kv[2 * i] * P[2 * i], kv[2 * i + 1] * P[2 * i + 1]);
          put16(reinterpret_cast<uint16_t*>(&ps.kdec[0][0]), w, pt);
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = Bf16::pack(vv[2 * i], vv[2 * i + 1]);
          put16(reinterpret_cast<uint16_t*>(&ps.vs[0][0]), w, pt);
        }
        po.gamma[kc] = P[15];
#pragma unroll
        for (int lv = 0; lv < 4; ++lv) {
          const int s = 8 >> lv;
          float ar[16], bc[8];  // this channel's row (k rows 0-7, q rows 8-15) and column operands
#pragma unroll
          for (int blk = 0; blk < 8 / s; ++blk) {
            const int m = blk * 2 * s + s;
            float f = 1.f;
#pragma unroll
            for (int i = m; i < m + s; ++i) {
              if (i > m) f *= al[i];
              const int r = blk * s + (i - m);
              ar[r] = DELTA ? kv[i] * f : 0.f;
              ar[8 + r] = qv[i] * f;
            }
            f = 1.f;
#pragma unroll
            for (int i = m - 1; i >= m - s; --i) {
              f *= al[i + 1];
              bc[blk * s + (i - (m - s))] = kv[i] * f;
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = QK::pack(ar[2 * i], ar[2 * i + 1]);
          put16(reinterpret_cast<uint16_t*>(&ps.A_lv[lv][0][0]), w, pt);
          *reinterpret_cast<uint4*>(&ps.B_lv[lv][pt][0]) =
              make_uint4(QK::pack(bc[0], bc[1]), QK::pack(bc[2], bc[3]), QK::pack(bc[4], bc[5]), QK::pack(bc[6], bc[7]));
        }
      }
      fence_proxy_async_smem();  // the reads of pin[buf] precede the next TMA write into it
      prep_bar();  // (D) tiles, level operands and norm partial sums written
      if (pt == 0 && !failed && c + 2 * kCtas < nch)  // (no new copy after a failed wait)
        issue_inputs(maps, sm.pin[buf], &sm.pinbar[buf], h, ts + (c + 2 * kCtas) * kChunk, p.gate_mode);
      // the norm factors of the 16 tokens (the partial sums are complete): lane
      // i < 16 of every warp holds token i's
      float rq_l = 1.f, rk_l = 1.f;
      if (L2N && lane < 16) {
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          sq += ps.red[w][lane];
          sk += ps.red[w][16 + lane];
        }
        rq_l = rsqrtf(sq + 1e-6f);
        rk_l = rsqrtf(sk + 1e-6f);
      }
      if (pw == 0 && lane < 16) po.sr[lane] = p.scale * rq_l;
      {  // level pw of the anchored split: raw L (rows 0-7, times beta) and Mqk (rows 8-15),
         // two accumulator chains, operands loaded one step ahead
        const int lv = pw;
        const int ls = 3 - lv;  // half-block size 2^ls = 8 >> lv
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // A^T and B^T are stored [channel][row]: .trans loads; lane matrix m of
        // A = (row half m & 1, channel half m >> 1)
        const int a_row = (lane >> 4) * 8 + (lane & 7), a_half = (lane >> 3) & 1;
        uint32_t a[2][4], b[2][2];
        ldsm_x4_trans(a[0], &ps.A_lv[lv][0][0] + cm_off(a_row, a_half));
        ldsm_x2_trans(b[0], &ps.B_lv[lv][lane & 15][0]);
#pragma unroll
        for (int kk = 0; kk < FD / 16; ++kk) {
          const int cur = kk & 1;
          if (kk + 1 < FD / 16) {
            ldsm_x4_trans(a[cur ^ 1], &ps.A_lv[lv][0][0] + cm_off(16 * (kk + 1) + a_row, a_half));
            ldsm_x2_trans(b[cur ^ 1], &ps.B_lv[lv][16 * (kk + 1) + (lane & 15)][0]);
          }
          mma16816<QK>(acc[cur], a[cur], b[cur][0], b[cur][1]);
        }
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = g + ((e & 2) ? 8 : 0);
          const int cidx = 2 * t + (e & 1);
          const int rr = r & 7;
          if ((rr >> ls) != (cidx >> ls)) continue;
          const int i = row_tok_f(ls, rr), jx = col_tok_f(ls, cidx);
          const float v = acc[0][e] + acc[1][e];
          if (r < 8) {
            if (DELTA) ps.Lm[i][jx] = ps.beta[jb][i] * v;
          } else {
            ps.Mq[i][jx] = v;
          }
        }
        if (pw == 0 && lane < 16)  // the diagonal of Mqk: q~_i . k~_i
          ps.Mq[lane][lane] = ps.red[0][32 + lane] + ps.red[1][32 + lane] + ps.red[2][32 + lane] + ps.red[3][32 + lane];
      }
      prep_bar();  // (E) raw L and Mqk complete
      if (pw == 0) {
        if (DELTA) {
          // X = -L = -diag(beta rk) raw diag(rk) in registers, then INV' forms
          const int g = lane >> 2, t = lane & 3;
          const float rkr[2] = {__shfl_sync(0xffffffffu, rk_l, g), __shfl_sync(0xffffffffu, rk_l, g + 8)};
          float rkc[2][2], bcol[2][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              rkc[nt][e] = __shfl_sync(0xffffffffu, rk_l, 8 * nt + 2 * t + e);
              bcol[nt][e] = ps.beta[jb][8 * nt + 2 * t + e];
            }
          Frag16 X;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              X.c[nt][e] = -ps.Lm[g + 8 * (e >> 1)][8 * nt + 2 * t + (e & 1)] * rkr[e >> 1] * rkc[nt][e & 1];
          const Frag16 inv = neumann_inverse16_frag<QK>(X, lane);
          Frag16 iw, ihi, ilo;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float u = inv.c[nt][e] * bcol[nt][e & 1] * rkr[e >> 1];  // INV_U
              iw.c[nt][e] = u * rkc[nt][e & 1];                                // INV_W
              ihi.c[nt][e] = __bfloat162float(__float2bfloat16_rn(u));
              ilo.c[nt][e] = u - ihi.c[nt][e];
            }
          uint32_t f[3][4];
          frag_as_a<QK>(iw, f[0]);
          frag_as_a<Bf16>(ihi, f[1]);
          frag_as_a<Bf16>(ilo, f[2]);
#pragma unroll
          for (int jj = 0; jj < 3; ++jj) ps.inv[lane][jj] = make_uint4(f[jj][0], f[jj][1], f[jj][2], f[jj][3]);
        }
      } else {
        // warps 1-3: Mqk~ into the slot. The level MMAs rewrite every strictly
        // lower entry of L and Mqk each chunk (each pair i > j belongs to exactly
        // one level) and the diagonal of Mqk is rewritten too, so the entries
        // never written stay at their initial zero: no clearing between chunks.
        for (int e = pt - 32; e < 256; e += 96) {
          const float x = ps.Mq[e >> 4][e & 15];
          const typename ST2::T v = ST2::cvt(x);
          po.mqk[e >> 4][e & 15] = *reinterpret_cast<const uint16_t*>(&v);
        }
        // and the group's next chunk's beta and gate into the other buffer
        if (c + 2 * kCtas < nch) {
          stage_next(jb ^ 1, c + 2 * kCtas);
          if (c + 4 * kCtas < nch) load_next(c + 4 * kCtas);
        }
      }
      prep_bar();  // (F) INV' fragments, Mqk~, the next chunk's beta
      if (DELTA) {
        uint32_t a[4], ahi[4], alo[4];
        {
          const uint4 x0 = ps.inv[lane][0], x1 = ps.inv[lane][1], x2 = ps.inv[lane][2];
          a[0] = x0.x; a[1] = x0.y; a[2] = x0.z; a[3] = x0.w;
          ahi[0] = x1.x; ahi[1] = x1.y; ahi[2] = x1.z; ahi[3] = x1.w;
          alo[0] = x2.x; alo[1] = x2.y; alo[2] = x2.z; alo[3] = x2.w;
        }
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int n0 = pw * 32 + 16 * pp;
          uint32_t b[4];
          ldsm_x4(b, &ps.kdec[0][0] + cm_off(n0 + (lane >> 4) * 8 + (lane & 7), (lane >> 3) & 1));
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816<QK>(c0, a, b[0], b[1]);
          mma16816<QK>(c1, a, b[2], b[3]);
          // -W' [tokens x keys n0 .. n0 + 15]: this lane's accumulators are its
          // B fragments of -W'^T in the recurrence (token tiles 0 and 1)
          po.W[n0 >> 4][lane] = make_uint4(Bf16::pack(-c0[0], -c0[1]), Bf16::pack(-c1[0], -c1[1]),
                                           Bf16::pack(-c0[2], -c0[3]), Bf16::pack(-c1[2], -c1[3]));
          // U~'^T [value rows n0 .. n0 + 15 x tokens] = v^T INV_U^T: A from the
          // channel-major v tile; the B fragments of INV_U^T are INV_U's A
          // fragments taken in another order (hi and lo parts)
          ldsm_x4(b, &ps.vs[0][0] + cm_off(n0 + ((lane >> 3) & 1) * 8 + (lane & 7), lane >> 4));
          float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816<Bf16>(u0, b, ahi[0], ahi[2]);
          mma16816<Bf16>(u0, b, alo[0], alo[2]);
          mma16816<Bf16>(u1, b, ahi[1], ahi[3]);
          mma16816<Bf16>(u1, b, alo[1], alo[3]);
          po.ut[n0 >> 4][0][lane] = make_float4(u0[0], u0[1], u0[2], u0[3]);
          po.ut[n0 >> 4][1][lane] = make_float4(u1[0], u1[1], u1[2], u1[3]);
        }
      } else {
        // delta rule off: U' = diag(rk) v, value channel pt of the 16 tokens
        float uv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) uv[i] = vv[i] * __shfl_sync(0xffffffffu, rk_l, i);
        // value row pt (row r of its 16-row tile) at token i sits in token tile
        // i / 8, lane 4 (r % 8) + (i % 8) / 2, entry 2 (r / 8) + i % 2
        float* ut = reinterpret_cast<float*>(&po.ut[pt >> 4][0][0]);
        const int r = pt & 15;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          ut[((i >> 3) * 32 + 4 * (r & 7) + ((i & 7) >> 1)) * 4 + 2 * (r >> 3) + (i & 1)] = uv[i];
      }
      prep_bar();  // (G) every store into the slot precedes the hand-off
      sig_pending = j;
    }
    signal_written();
  } else if (warp == kMoverWarp) {
    // ===================== mover warp =====================
    // Loads chunk c from its global slot into local stage c mod kRing once the
    // slot is published and the recurrence warps have released the stage; a
    // released stage also returns its chunk's global slot to the producer.
    if (lane == 0) {
      bool failed = false;
      int last_issued = -1;
      for (int c = 0; c < nch; ++c) {
        const int s = c & (kRing - 1);
        const int gs = c % kGRing;
        if (c >= kRing) {
          if (!failed && !mbar_wait_bounded(smem_u32(&sm.empty[s]), static_cast<uint32_t>(c / kRing - 1) & 1u,
                                            kWaitLimitNs)) {
            failed = true;
            set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
          }
          const int cp = c - kRing;
          mbar_arrive_cluster(mapa_shared(smem_u32(&sm.gfree[cp % kGRing]), static_cast<uint32_t>(cp % kCtas)));
        }
        if (!failed && !mbar_wait_acq_cluster_bounded(smem_u32(&sm.ready[gs]), static_cast<uint32_t>(c / kGRing) & 1u,
                                                      kWaitLimitNs)) {
          failed = true;
          set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
        }
        if (failed) continue;  // after a failed wait no new copy is started
        fence_proxy_async_global();  // the bulk loads below read what the acquire made visible
        const unsigned char* slot = gring + static_cast<size_t>(gs) * kSlotBytes;
        unsigned char* stage = reinterpret_cast<unsigned char*>(&sm.ring[s]);
        mbar_arrive_expect_tx_local(&sm.full[s], kStageTx);
        bulk_load_g2s(stage, slot, kSharedBytes, &sm.full[s]);
        bulk_load_g2s(stage + kSharedBytes, slot + kSharedBytes + rank * kUtSliceBytes, kUtSliceBytes, &sm.full[s]);
        last_issued = c;
      }
      // no load may still be landing in this CTA's shared memory when it exits:
      // the last stages' copies are waited for (bounded) even after a failure
      for (int c = max(0, last_issued - kRing + 1); c <= last_issued; ++c)
        if (!mbar_wait_bounded(smem_u32(&sm.full[c & (kRing - 1)]), static_cast<uint32_t>(c / kRing) & 1u,
                               kWaitLimitNs))
          set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
    }
    __syncwarp();
  } else if (warp == kPublisherWarp) {
    // ===================== publisher warp =====================
    // Publishes each chunk the prep groups wrote into the global ring: lanes
    // 0-3 each make the group's stores visible at cluster scope and arrive on
    // the slot's "ready" mbarrier in CTA `lane`.
    bool failed = false;
    for (int j = 0, c = static_cast<int>(rank); c < nch; ++j, c += kCtas) {
      if (lane < kCtas) {
        if (!failed && !mbar_wait_bounded(smem_u32(&sm.sig[j % (kGRing / kCtas)]),
                                          static_cast<uint32_t>(j / (kGRing / kCtas)) & 1u, kWaitLimitNs)) {
          failed = true;
          set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
        }
        fence_acq_rel_cluster();
        mbar_arrive_relaxed_cluster(mapa_shared(smem_u32(&sm.ready[c % kGRing]), static_cast<uint32_t>(lane)));
      }
      __syncwarp();
    }
  } else if (warp == kOutputWarp) {
    // ===================== output warp =====================
    // Stores each chunk's 16 x 32 block of o (lane: one token, 16 value rows)
    // from the staged O and releases the stage.
    const int tok = lane >> 1, hv = lane & 1;
    bool failed = false;
    for (int c = 0; c < nch; ++c) {
      const int s = c & (kRing - 1);
      if (!failed &&
          !mbar_wait_bounded(smem_u32(&sm.ofull[s]), static_cast<uint32_t>(c / kRing) & 1u, kWaitLimitNs)) {
        failed = true;
        if (lane == 0) set_err(p.err, 4 /* KDA_ERR_TIMEOUT */);
      }
      const float* p0 = &sm.rs.opart[s][tok][hv * 16];
      const float sr = sm.ring[s].sr[tok];  // scale rq of the token (the stage is held until the release below)
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(p0 + 4 * i);
        pk[2 * i] = Bf16::pack(sr * x.x, sr * x.y);
        pk[2 * i + 1] = Bf16::pack(sr * x.z, sr * x.w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_local(&sm.empty[s]);
      const int tok0 = ts + c * kChunk;
      if (tok < te - tok0) {  // rows past the sequence end belong to the next sequence
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                              (static_cast<size_t>(tok0 + tok) * H + h) * FD + rank * kRows + hv * 16);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
  }
  cluster_sync_all();
  if (rank == 0 && tid == 0 && ring_id >= 0) {  // hand the ring back to the pool
    __threadfence();
    atomicAnd(reinterpret_cast<unsigned int*>(p.records) + ring_id / 32, ~(1u << (ring_id % 32)));
  }
}

// The workspace holds kPool rings and every resident cluster holds one, so at
// most kPool clusters of the kernel may be resident at once (a cluster that
// found no free ring would wait out its bounded claim and report a timeout).
// Checked once per device with the occupancy calculator; a device that could
// hold more is refused with cudaErrorNotSupported (KDA_ERR_UNSUPPORTED).
template <typename Kernel>
cudaError_t check_cluster_residency_once(Kernel kernel, size_t smem, std::atomic<uint64_t>& ok_devs,
                                         std::atomic<uint64_t>& bad_devs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (ok_devs.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  if (bit != 0 && (bad_devs.load(std::memory_order_acquire) & bit) != 0) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCtas * 64, 1, 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;  // the cluster shape is the kernel's compile-time one
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters > kPool) {
    bad_devs.fetch_or(bit, std::memory_order_acq_rel);
    return cudaErrorNotSupported;
  }
  ok_devs.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <bool DELTA, bool L2N, int MODE>
cudaError_t launch_fused_t(const ChunkCall& c, cudaStream_t s) {
  using QK = std::conditional_t<L2N, F16, Bf16>;
  const size_t smem = sizeof(FusedSmem<typename QK::T, MODE>);
  static std::atomic<uint64_t> smem_set{0}, resident_ok{0}, resident_bad{0};
  {
    cudaError_t e = set_smem_limit_once(kda_chunk_fused_kernel<DELTA, L2N, MODE>, smem, smem_set);
    if (e != cudaSuccess) return e;
    e = check_cluster_residency_once(kda_chunk_fused_kernel<DELTA, L2N, MODE>, smem, resident_ok, resident_bad);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = static_cast<unsigned>(c.geo.N) * static_cast<unsigned>(c.geo.H) * kCtas;
  if (grid == 0) return cudaSuccess;
  TmaInputMaps maps;
  cudaError_t e = encode_input_maps(c, &maps);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(c.records, 0, kPoolHeader, s);  // every pool ring free
  if (e != cudaSuccess) return e;
  kda_chunk_fused_kernel<DELTA, L2N, MODE><<<grid, kFusedThreads, smem, s>>>(c, maps);
  return cudaGetLastError();
}

}  // namespace

static_assert(sizeof(FusedSmem<__half, 0>) <= 227 * 1024 && sizeof(FusedSmem<__nv_bfloat16, 0>) <= 227 * 1024 &&
                  sizeof(FusedSmem<__half, 2>) <= 227 * 1024 && sizeof(FusedSmem<__nv_bfloat16, 2>) <= 227 * 1024,
              "fused kernel shared memory");

size_t fused_workspace_bytes() { return kPoolHeader + static_cast<size_t>(kPool) * kRingBytes; }

template <int MODE>
cudaError_t launch_fused_mode(const ChunkCall& c, cudaStream_t s) {
  if (c.delta) return c.l2norm ? launch_fused_t<true, true, MODE>(c, s) : launch_fused_t<true, false, MODE>(c, s);
  return c.l2norm ? launch_fused_t<false, true, MODE>(c, s) : launch_fused_t<false, false, MODE>(c, s);
}

cudaError_t launch_chunk_fused(const ChunkCall& c, cudaStream_t s) {
  if (c.dk != FD || c.dv != FD) return cudaErrorInvalidValue;
  if (c.output_pass) return c.h_chunks != nullptr ? launch_fused_mode<2>(c, s) : cudaErrorInvalidValue;
  return c.h_chunks != nullptr ? launch_fused_mode<1>(c, s) : launch_fused_mode<0>(c, s);
}

}  // namespace kda
