/*
 * kda.h - C ABI of the GB300 (sm_103a) Kimi Delta Attention library (libkda.so).
 *
 * Operations
 *   kda_chunk_fwd             chunkwise KDA forward over one batch of sequences
 *   kda_chunk_workspace_size  scratch bytes kda_chunk_fwd needs for given arguments
 *   kda_chunk_output          chunk-parallel output pass from per-chunk entering states
 *   kda_decode_step           fused T=1 decode step on a packed q|k|v row with a slot pool
 *   kda_decode_conv_step      the decode step with its causal conv1d + SiLU fused in front
 *   kda_recurrent_step        T tokens per row (T <= 64) on a slot pool: speculative / extend steps
 *   kda_head_rmsnorm          output-side per-head RMSNorm of attention outputs
 *   kda_chunk_fwd_noalloc     kda_chunk_fwd on a library-owned scratch buffer (no allocation)
 *   kda_version               library version string
 *   kda_selftest_*            diagnostics: bounded-wait failure path, tcgen05 round trip
 *
 * What is computed (per sequence n and head h; math state S is [dk, dv], stored
 * transposed as [dv, dk] with dk contiguous):
 *   S~  = diag(e^{g_t}) S                        decay on the key index
 *   u_t = beta_t (v_t - S~^T k_t)                delta rule (u_t = v_t with KDA_FLAG_DELTA_OFF)
 *   S   = S~ + k_t u_t^T
 *   o_t = scale S^T q_t
 * ("TileLang 实战：KDA 从零到一" §1 gives this recurrence in the transposed
 * (d_v, d_k) form; "FlashKDA里的L矩阵和Mqk矩阵" §背景 gives the same token
 * recurrence in delta form.) kda_chunk_fwd evaluates it in 16-token chunks
 * through the per-chunk L matrix, the Mqk matrix, the exact Neumann inverse of
 * (I + L) and a serial cross-chunk state recurrence (the same page, sections
 * L矩阵的构造, Mqk矩阵的构造, 为什么CHUNK=16, K2 内核如何消费).
 *
 * Conventions shared by every call
 *   - All tensor pointers are caller-owned DEVICE memory, contiguous row-major,
 *     16-byte aligned. The library never allocates, frees or synchronises.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Argument errors are detected on the host before any launch and return
 *     KDA_ERR_INVALID_ARG or KDA_ERR_UNSUPPORTED; nothing is launched then.
 *   - A failed launch returns KDA_ERR_CUDA.
 *   - Problems only visible on the device (a bad cu_seqlens array, an
 *     out-of-range slot index, a bounded wait that ran out) are written as a
 *     kda_status code into the optional device word `err` (if non-NULL); the
 *     affected work is skipped. `err` is never cleared by the library.
 *   - Not thread-safe per stream in any special way: calls on one stream run
 *     in order; concurrent calls on different streams must not share outputs
 *     or workspace.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, bad index array */
  KDA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (e.g. dk = 96) */
  KDA_ERR_CUDA = 3,         /* a CUDA launch or runtime call failed */
  KDA_ERR_TIMEOUT = 4,      /* a bounded device-side wait expired (reported through err) */
  KDA_ERR_TOO_LARGE = 5     /* needs more scratch than kda_chunk_fwd_noalloc's fixed buffer */
} kda_status;

typedef enum {
  KDA_DTYPE_BF16 = 0,  /* q, k, v, beta/b and o in bfloat16; tensor-core path */
  KDA_DTYPE_FP32 = 1   /* q, k, v, beta/b and o in float32; CUDA-core fp32 path */
} kda_dtype;

typedef enum {
  KDA_GATE_NONE = 0,    /* g = 0 (no decay) */
  KDA_GATE_G = 1,       /* log-decay g given: fp32 [B, T, H, dk] */
  KDA_GATE_INPUTS = 2,  /* g = -exp(A_log[h]) * softplus(a + dt_bias) computed in the kernel */
  KDA_GATE_HEAD_G = 3   /* Gated DeltaNet: one log-decay per token and head, g fp32 [B, T, H],
                           applied to every key channel (TileLang 实战 §1 ladder) */
} kda_gate_mode;

typedef enum {
  KDA_BETA_VALUES = 0,  /* beta given: [B, T, H] in the input dtype */
  KDA_BETA_LOGITS = 1   /* logits b given: beta = sigmoid(b), [B, T, H] in the input dtype */
} kda_beta_mode;

/* flags */
#define KDA_FLAG_L2NORM_QK 0x1u  /* q <- q / sqrt(sum q^2 + 1e-6), same for k, in the kernel */
#define KDA_FLAG_DELTA_OFF 0x2u  /* u_t = v_t: plain (gated) linear attention, beta ignored */
/* Debug (decode, decode-conv and recurrent steps): before the step, check that
 * the valid slot indices are distinct; a repeat writes KDA_ERR_INVALID_ARG to
 * err (which the flag requires). The step itself still runs: the check
 * reports a caller error, it does not repair it. O(B^2) work. */
#define KDA_FLAG_CHECK_INDICES 0x4u

/*
 * Arguments of kda_chunk_fwd.
 *
 * Shapes (row-major, contiguous):
 *   q, k      [B, T, H, dk]        dtype
 *   v, o      [B, T, H, dv]        dtype
 *   g         [B, T, H, dk]        fp32   (KDA_GATE_G), or [B, T, H] (KDA_GATE_HEAD_G)
 *   a         [B, T, H*dk]         fp32   (KDA_GATE_INPUTS)
 *   A_log     [H]                  fp32   (KDA_GATE_INPUTS)
 *   dt_bias   [H*dk]               fp32   (KDA_GATE_INPUTS)
 *   beta      [B, T, H]            dtype  (values or logits, per beta_mode)
 *   h0, hT    [N, H, dv, dk]       fp32   (either may be NULL: zero initial state /
 *                                          no final state)
 *   cu_seqlens [N + 1]             int32  device array, or NULL
 * Without cu_seqlens the batch holds N = B independent sequences of length T.
 * With cu_seqlens, B must be 1 and the N sequences are packed along T:
 * sequence n spans tokens [cu_seqlens[n], cu_seqlens[n+1]). cu_seqlens must
 * start at 0, never decrease and end at T; this is checked on the device and a
 * violation writes KDA_ERR_INVALID_ARG to err and skips the call's work.
 * Chunks of 16 tokens restart at every sequence start.
 * Supported: dtype BF16 with dk = dv in {64, 128}; dtype FP32 with dk, dv in {64, 128}.
 * Numerics of the BF16 path: S stays fp32 on chip; the contractions run on
 * tensor cores with fp32 accumulation, S rounded to bf16 as an operand, and
 * (with the delta rule on) the corrected values U in fp16, which assumes
 * |U| < 65504 (values are saturated, never turned into inf, and no status is
 * reported). With KDA_FLAG_L2NORM_QK and dk = dv = 128 the operand held in fp16
 * is U / |k~| (k~ the token's key before the norm), so the bound applies to
 * that scaled value there.
 */
typedef struct kda_chunk_args {
  int32_t dtype;       /* kda_dtype */
  int32_t B, T, H, dk, dv;
  int32_t N;           /* number of sequences (B without cu_seqlens) */
  int32_t gate_mode;   /* kda_gate_mode */
  int32_t beta_mode;   /* kda_beta_mode; ignored with KDA_FLAG_DELTA_OFF */
  uint32_t flags;      /* KDA_FLAG_* */
  float scale;         /* output scale, typically dk^-0.5 */
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* a;
  const float* A_log;
  const float* dt_bias;
  const void* beta;
  const float* h0;
  const int32_t* cu_seqlens;
  void* o;
  float* hT;
  int32_t* err;        /* optional device status word */
  float* h_chunks;     /* optional per-chunk entering states (see below), or NULL */
} kda_chunk_args;

/*
 * Per-chunk entering states (h_chunks). When non-NULL, kda_chunk_fwd also
 * writes the state entering every 16-token chunk: fp32 [C_total, H, dv, dk],
 * chunk by chunk in sequence order (uniform batches: B * ceil(T/16) entries,
 * chunk c of sequence n at n * ceil(T/16) + c; with cu_seqlens: the sum over
 * sequences of ceil(len/16), each sequence's chunks after the previous
 * sequence's). Entry 0 of a sequence is its h0 (or zeros). These are the
 * materialised states of the chunkwise form that a chunk-parallel output pass
 * (kda_chunk_output) and a backward pass start from. bf16 only. With
 * dk = dv = 128 the fused kernel writes them as it goes (streaming stores of
 * the state its recurrence holds); d = 64 runs the two-kernel path.
 */

/*
 * Bytes of device scratch memory kda_chunk_fwd needs for these arguments
 * (0 when the arguments are invalid). The workspace is caller-owned; its
 * contents on entry do not matter and are garbage on exit. For bf16 with
 * dk = dv = 128 it is a fixed ~14 MB (a pool of L2-resident rings through
 * which the kernel hands prepared chunks between the CTAs of a cluster) plus a
 * small per-sequence header; other shapes need per-(chunk, head) records.
 * kda_chunk_output needs the same scratch as kda_chunk_fwd for the same
 * arguments.
 */
size_t kda_chunk_workspace_size(const kda_chunk_args* args);

/*
 * Chunkwise KDA forward. Writes o (and hT when non-NULL). `workspace` is device
 * memory of at least kda_chunk_workspace_size(args) bytes, 256-byte aligned.
 * Returns KDA_OK once the work is enqueued. For bf16 with dk = dv = 128 the
 * first call on a device also checks that the device cannot hold more of the
 * fused kernel's 4-CTA clusters at once than the workspace has rings (40; a
 * GB300 holds 38) and returns KDA_ERR_UNSUPPORTED, launching nothing, where it
 * could.
 */
kda_status kda_chunk_fwd(const kda_chunk_args* args, void* workspace, size_t workspace_bytes,
                         kda_stream_t stream);

/*
 * Chunk-parallel output pass: o from the inputs and the per-chunk entering
 * states args->h_chunks (read, as kda_chunk_fwd writes them). Every chunk's
 * output o_c = q_dec,c S_c + Mqk_c U_c, U_c = U~_c - W_c S_c, is formed
 * independently of the others (the serial dependence lives in the states).
 * Same arguments, workspace and layouts as kda_chunk_fwd; h0 and hT are
 * ignored; bf16 only, h_chunks required (KDA_ERR_INVALID_ARG otherwise).
 */
kda_status kda_chunk_output(const kda_chunk_args* args, void* workspace, size_t workspace_bytes,
                            kda_stream_t stream);

/*
 * Arguments of kda_decode_step (sglang PR #26586, fused_recurrent_kda_packed_decode:
 * one token per batch row, read from a packed [q | k | v] row).
 *
 *   packed_qkv [B, 2*H*K + HV*V]   bf16  row = [q (H*K) | k (H*K) | v (HV*V)]
 *   a          [B, HV*K]           bf16  gate input
 *   b          [B, HV]             bf16  beta logits (beta = sigmoid(b))
 *   A_log      [HV]                fp32
 *   dt_bias    [HV*K]              fp32
 *   state_pool [num_slots, HV, V, K] fp32, updated IN PLACE for the valid rows
 *   indices    [B]                 int32 slot of each row; negative = padding row
 *   o          [B, HV, V]          bf16
 * Value head hv uses query/key head hv / (HV / H); HV must be a multiple of H.
 * g = -exp(A_log[hv]) * softplus(a + dt_bias); with KDA_FLAG_L2NORM_QK q and k
 * are L2-normalised (eps 1e-6 inside the root); q is multiplied by scale.
 * A padding row writes o = 0 and touches no state. Valid indices must be
 * distinct (rows sharing a slot race; KDA_FLAG_CHECK_INDICES checks it). An
 * index >= num_slots writes KDA_ERR_INVALID_ARG to err, zeroes that row's o
 * and touches no state.
 * Supported: K, V in {64, 128}.
 */
typedef struct kda_decode_args {
  int32_t B, H, HV, K, V;
  int32_t num_slots;
  uint32_t flags;      /* KDA_FLAG_L2NORM_QK, KDA_FLAG_CHECK_INDICES */
  float scale;
  const void* packed_qkv;
  const void* a;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  const int32_t* indices;
  void* o;
  int32_t* err;        /* optional device status word */
} kda_decode_args;

/* Fused T=1 decode step. Returns KDA_OK once the work is enqueued. */
kda_status kda_decode_step(const kda_decode_args* args, kda_stream_t stream);

/*
 * The decode step with its depthwise causal conv1d + SiLU fused in front (the
 * sglang PR #26586 summary's KDAAttnBackend.forward_decode runs
 * causal_conv1d_update(mixed_qkv, conv_states, conv_weights, bias,
 * activation="silu") right before the packed decode). For every valid row b
 * with slot s and every channel c of the packed row (C = 2*H*K + HV*V):
 *   window = [conv_state_in[s, 0..W-2, c], dec.packed_qkv[b, c]]   (oldest first)
 *   x[b, c] = silu(sum_i conv_weight[c, i] * window[i] + conv_bias[c])
 *   conv_state_out[s, :, c] = window[1..W-1]
 * then the decode step of kda_decode_step runs on x as its packed q|k|v row.
 *   dec             all fields as for kda_decode_step; dec.packed_qkv holds
 *                   the conv input (bf16 [B, C])
 *   W               conv width, 2..4
 *   conv_state_in   bf16 [num_slots, W-1, C]
 *   conv_state_out  bf16 [num_slots, W-1, C]; only the valid rows' slots are
 *                   written. It may be conv_state_in (update in place) only
 *                   when HV == H: with HV > H a q/k channel is read by the HV/H
 *                   value heads of its group and written by the first one, so
 *                   an in-place update would race.
 *   conv_weight     fp32 [C, W] (tap W-1 multiplies the newest input)
 *   conv_bias       fp32 [C] or NULL
 * Padding rows write o = 0 and touch neither pool. Returns KDA_OK once the
 * work is enqueued.
 */
typedef struct kda_decode_conv_args {
  kda_decode_args dec;
  int32_t W;
  const void* conv_state_in;
  void* conv_state_out;
  const float* conv_weight;
  const float* conv_bias;
} kda_decode_conv_args;
kda_status kda_decode_conv_step(const kda_decode_conv_args* args, kda_stream_t stream);

/*
 * Arguments of kda_recurrent_step: T tokens per batch row on a state-slot pool.
 * This is the general fused recurrent step that the packed decode specialises
 * (sglang PR #26586 summary, 功能与动机 and 实现拆解: the packed kernel takes over
 * the generic path for one token per row); several tokens per row occur in
 * speculative and extend steps.
 *
 *   q, k       [B, T, H, K]          bf16
 *   v          [B, T, HV, V]         bf16
 *   a          [B, T, HV*K]          bf16  gate input
 *   b          [B, T, HV]            bf16  beta logits (beta = sigmoid(b))
 *   A_log      [HV]                  fp32
 *   dt_bias    [HV*K]                fp32
 *   state_pool [num_slots, HV, V, K] fp32, updated IN PLACE for the valid rows
 *   indices    [B]                   int32 slot of each row; negative = padding row
 *   o          [B, T, HV, V]         bf16
 * The T tokens of a row are applied to its slot's state in order. Everything
 * else is as for kda_decode_step: value head hv uses query/key head
 * hv / (HV / H); the gate, beta, L2 norm (KDA_FLAG_L2NORM_QK) and scaling of q;
 * a padding row writes o = 0 for all its tokens and touches no state; valid
 * indices must be distinct; an index >= num_slots writes KDA_ERR_INVALID_ARG
 * to err, zeroes that row's o and touches no state.
 * Supported: K, V in {64, 128}; 1 <= T <= KDA_RECURRENT_MAX_T (longer
 * sequences belong to kda_chunk_fwd). q, k, v, a, dt_bias, state_pool and o
 * must be 16-byte aligned.
 * Resources: with K = 128 and T > 16 each CTA (one per row and value head)
 * holds V columns of tensor memory while it runs, at most four CTAs per SM.
 * A kernel on another stream that holds tensor memory on the same SMs at the
 * same time only delays this one's CTAs (their allocation waits); nothing is
 * left allocated when the call completes.
 */
#define KDA_RECURRENT_MAX_T 64
typedef struct kda_recurrent_args {
  int32_t B, T, H, HV, K, V;
  int32_t num_slots;
  uint32_t flags;      /* KDA_FLAG_L2NORM_QK, KDA_FLAG_CHECK_INDICES */
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const void* a;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  const int32_t* indices;
  void* o;
  int32_t* err;        /* optional device status word */
} kda_recurrent_args;

/* Short-T recurrent step. Returns KDA_OK once the work is enqueued. */
kda_status kda_recurrent_step(const kda_recurrent_args* args, kda_stream_t stream);

/*
 * Output-side per-head RMSNorm ("06 · linear 路线（一）" §1 and §4 (3): GLA, GDN
 * and KDA drop the linear-attention normaliser and normalise each head's
 * output instead). The pages give no formula; this is the plain RMSNorm:
 *   y[r, :] = x[r, :] / sqrt(mean(x[r, :]^2) + eps) * weight[:]
 * over R rows of V values, a row being one token of one head (o of the chunk
 * forward or the decode viewed as [B*T*H, V]).
 *   x, y    [R, V]   bf16, 16-byte aligned; y may be x (in place)
 *   weight  [V]      fp32, 16-byte aligned
 * Supported: V in {64, 128}. Returns KDA_OK once the work is enqueued.
 */
typedef struct kda_rmsnorm_args {
  int64_t R;
  int32_t V;
  float eps;
  const void* x;
  const float* weight;
  void* y;
} kda_rmsnorm_args;
kda_status kda_head_rmsnorm(const kda_rmsnorm_args* args, kda_stream_t stream);

/*
 * Chunk forward for callers that cannot allocate device memory.
 *
 * No counterpart in the method's description: this is a deployment aid. Some
 * callers may not call cudaMalloc (or any allocating routine) at the point
 * where they run the attention: code recording a CUDA graph or replaying a
 * fixed memory plan, runtimes that hand out every device byte at start-up and
 * forbid allocation afterwards, and bindings with no device allocator of their
 * own. kda_chunk_fwd needs a caller-provided workspace; this entry point uses
 * instead a scratch buffer of KDA_NOALLOC_SCRATCH_BYTES that the library owns:
 * a file-scope __device__ array, present on every GPU that loads the library
 * until the process exits.
 *
 * Arguments and results are those of kda_chunk_fwd; inputs and outputs are
 * still caller-owned device memory. The call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine).
 *
 * Returns KDA_ERR_TOO_LARGE, launching nothing, when the arguments need more
 * than KDA_NOALLOC_SCRATCH_BYTES of scratch (kda_chunk_workspace_size(args)
 * tells how much they need; bf16 with dk = dv = 128 needs a fixed ~14 MB plus
 * 4 bytes per sequence). Other argument errors as for kda_chunk_fwd.
 *
 * The first call on each device looks up the address of the device's copy of
 * the buffer (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture. Later calls only read the cached address.
 * The buffer's contents on entry do not matter (every byte a call reads is
 * written earlier in the same call), and it keeps the last call's contents.
 * All calls on a device share the one buffer: calls whose GPU work overlaps
 * (different streams, or other threads) race and corrupt each other; order
 * them on one stream or synchronise between them.
 * The looked-up address is kept for the life of the process: do not use this
 * entry point on a device after cudaDeviceReset (or any other destruction of
 * its primary context) in the same process.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20) /* 16 MiB */
kda_status kda_chunk_fwd_noalloc(const kda_chunk_args* args, kda_stream_t stream);

/* Version string of the library, e.g. "kda-gb300 0.1.0 sm_103a". */
const char* kda_version(void);

/*
 * Diagnostic: exercises the bounded device-side wait that every mbarrier wait
 * of the fused chunk kernel uses. One thread waits on a shared-memory mbarrier
 * that nothing arrives on, gives up after limit_ns nanoseconds (1e3 .. 1e10)
 * and writes KDA_ERR_TIMEOUT to *err (device int32, 4-byte aligned); the
 * kernel then returns and the context stays usable. Tests use it to check the
 * failure path without a fault or a hang.
 */
kda_status kda_selftest_bounded_wait(int32_t* err, uint64_t limit_ns, kda_stream_t stream);

/*
 * Diagnostic: one MMA of the 5th-generation tensor cores (tcgen05.mma,
 * kind::f16, bf16 operands, fp32 accumulator in tensor memory) and its round
 * trip. The method's pages have no counterpart; the chunk kernels use
 * warp-level mma.sync, and this call measures what the tensor-memory path
 * would cost them.
 *
 * One CTA computes d [128 x N] (fp32, row-major) = a [128 x K] * b^T, with a
 * and b bf16 row-major device arrays ([128, K] and [N, K]). The operands are
 * placed in shared memory in a K-major layout (no swizzle, or the 128-byte
 * swizzle), A optionally copied on into tensor memory (a_from_tmem) and read
 * from there; the result is read back with tcgen05.ld. Then `reps` round trips
 * (issue -> commit seen on an mbarrier -> the first 16 columns in registers)
 * are timed one by one, and `reps` MMA groups back to back under one commit.
 *
 * cycles (device int64[7], nullable) receives: [0] summed SM cycles from issue
 * to the completion being seen, [1] summed cycles from issue to the data in
 * registers, [2] cycles of the back-to-back burst (every group on the same
 * accumulator), [3] reps, [4] cycles of a second burst of `reps` groups that
 * rotates over [5] independent accumulators (0 when N leaves room for one),
 * [6] cycles the issuing thread took to issue the first burst.
 * K is 16, 32, 64 or 128; N a multiple of 16 in 16..256; layout 0 (none) or
 * 1 (128-byte swizzle); 0 <= reps <= 4096. Pointers 16-byte aligned (err:
 * 4-byte, may be NULL). Every wait is bounded: a wait that runs out writes
 * KDA_ERR_TIMEOUT to *err and the kernel returns after freeing its tensor
 * memory. Uses all of one SM's tensor memory while it runs.
 */
typedef struct kda_tcgen05_probe_args {
  int32_t K, N, layout, a_from_tmem, reps;
  const void* a;       /* bf16 [128, K] */
  const void* b;       /* bf16 [N, K] */
  float* d;            /* fp32 [128, N], written */
  long long* cycles;   /* int64 [7] or NULL */
  int32_t* err;        /* or NULL */
} kda_tcgen05_probe_args;
kda_status kda_selftest_tcgen05(const kda_tcgen05_probe_args* args, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
