// Host side of the C ABI declared in include/kda.h: argument validation,
// workspace layout and kernel dispatch. No allocation, no synchronisation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool chunk_dims_supported(const kda_chunk_args& a) {
  if (a.dtype == KDA_DTYPE_BF16) return a.dk == a.dv && (a.dk == 64 || a.dk == 128);
  if (a.dtype == KDA_DTYPE_FP32) return (a.dk == 64 || a.dk == 128) && (a.dv == 64 || a.dv == 128);
  return false;
}

// bf16 with dk = dv = 128 runs the fused cluster kernel (prep and recurrence in
// one launch; it also writes per-chunk states when asked, and forms the
// chunk-parallel output pass from them); other shapes run the two-kernel path
// through workspace records.
bool uses_fused(const kda_chunk_args& a) {
  return a.dtype == KDA_DTYPE_BF16 && a.dk == 128 && a.dv == 128;
}

// Returns KDA_OK and fills geometry when the arguments are well formed.
kda_status check_chunk(const kda_chunk_args* a, kda::ChunkGeom* geo, size_t* rec_bytes) {
  if (a == nullptr) return KDA_ERR_INVALID_ARG;
  if (a->dtype != KDA_DTYPE_BF16 && a->dtype != KDA_DTYPE_FP32) return KDA_ERR_INVALID_ARG;
  if (a->B < 1 || a->T < 0 || a->H < 1 || a->dk < 1 || a->dv < 1 || a->N < 1) return KDA_ERR_INVALID_ARG;
  if (a->flags & ~(KDA_FLAG_L2NORM_QK | KDA_FLAG_DELTA_OFF)) return KDA_ERR_INVALID_ARG;
  if (a->gate_mode < KDA_GATE_NONE || a->gate_mode > KDA_GATE_HEAD_G) return KDA_ERR_INVALID_ARG;
  const bool delta = !(a->flags & KDA_FLAG_DELTA_OFF);
  if (delta && a->beta_mode != KDA_BETA_VALUES && a->beta_mode != KDA_BETA_LOGITS) return KDA_ERR_INVALID_ARG;
  if (a->cu_seqlens == nullptr) {
    if (a->N != a->B) return KDA_ERR_INVALID_ARG;
  } else {
    if (a->B != 1) return KDA_ERR_INVALID_ARG;
    if (!aligned(a->cu_seqlens, 4)) return KDA_ERR_INVALID_ARG;
  }
  const int64_t tokens = static_cast<int64_t>(a->B) * a->T;
  if (tokens * a->H * (a->dk > a->dv ? a->dk : a->dv) > INT64_C(1) << 40) return KDA_ERR_INVALID_ARG;
  if (tokens > INT32_MAX / 2) return KDA_ERR_INVALID_ARG;
  if (!chunk_dims_supported(*a)) return KDA_ERR_UNSUPPORTED;
  if (a->h_chunks != nullptr) {  // per-chunk states: the bf16 two-kernel path only
    if (a->dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;
    if (!aligned(a->h_chunks, 16)) return KDA_ERR_INVALID_ARG;
  }
  if (tokens > 0) {
    if (!a->q || !a->k || !a->v || !a->o) return KDA_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16)) return KDA_ERR_INVALID_ARG;
    if (a->gate_mode == KDA_GATE_G && (!a->g || !aligned(a->g, 16))) return KDA_ERR_INVALID_ARG;
    if (a->gate_mode == KDA_GATE_HEAD_G && (!a->g || !aligned(a->g, 4))) return KDA_ERR_INVALID_ARG;
    if (a->gate_mode == KDA_GATE_INPUTS) {
      if (!a->a || !a->A_log || !a->dt_bias) return KDA_ERR_INVALID_ARG;
      if (!aligned(a->a, 16) || !aligned(a->A_log, 4) || !aligned(a->dt_bias, 4)) return KDA_ERR_INVALID_ARG;
    }
    if (delta) {
      const size_t el = a->dtype == KDA_DTYPE_BF16 ? 2 : 4;
      if (!a->beta || !aligned(a->beta, el)) return KDA_ERR_INVALID_ARG;
    }
  }
  if (a->h0 && !aligned(a->h0, 16)) return KDA_ERR_INVALID_ARG;
  if (a->hT && !aligned(a->hT, 16)) return KDA_ERR_INVALID_ARG;
  if (a->err && !aligned(a->err, 4)) return KDA_ERR_INVALID_ARG;

  geo->N = a->N;
  geo->T = a->T;
  geo->H = a->H;
  geo->cu_seqlens = a->cu_seqlens;
  geo->chunk_off = nullptr;
  geo->chunks_per_seq = (a->T + 15) / 16;
  if (a->cu_seqlens == nullptr) {
    geo->max_chunks = a->B * geo->chunks_per_seq;
  } else {
    geo->max_chunks = geo->chunks_per_seq + a->N;  // each sequence adds at most one partial chunk
  }
  *rec_bytes = a->dtype == KDA_DTYPE_BF16 ? kda::record_bytes_tc(a->dk) : kda::record_bytes_f32(a->dk, a->dv);
  if (*rec_bytes == 0) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

// Scratch of a call (kda_chunk_fwd and kda_chunk_output alike): the fused
// kernel's fixed pool of rings, or one record per (chunk, head) for the
// two-kernel path.
size_t workspace_bytes(const kda_chunk_args& a, const kda::ChunkGeom& geo, size_t rec_bytes) {
  if (uses_fused(a)) return kda::plan_header_bytes(geo.N) + kda::fused_workspace_bytes();
  return kda::plan_header_bytes(geo.N) + static_cast<size_t>(geo.max_chunks) * geo.H * rec_bytes;
}

}  // namespace

extern "C" {

size_t kda_chunk_workspace_size(const kda_chunk_args* args) {
  kda::ChunkGeom geo;
  size_t rec = 0;
  if (check_chunk(args, &geo, &rec) != KDA_OK) return 0;
  return workspace_bytes(*args, geo, rec);
}

namespace {

kda_status run_chunk(const kda_chunk_args* args, void* workspace, size_t ws_bytes, kda_stream_t stream,
                     bool output_pass) {
  kda::ChunkGeom geo;
  size_t rec = 0;
  kda_status st = check_chunk(args, &geo, &rec);
  if (st != KDA_OK) return st;
  if (output_pass && args->h_chunks == nullptr) return KDA_ERR_INVALID_ARG;
  const size_t need = workspace_bytes(*args, geo, rec);
  if (workspace == nullptr || ws_bytes < need || !aligned(workspace, 256)) return KDA_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  kda::ChunkCall c;
  c.geo = geo;
  c.geo.chunk_off = static_cast<int32_t*>(workspace);
  c.dk = args->dk;
  c.dv = args->dv;
  c.gate_mode = args->gate_mode;
  c.beta_mode = args->beta_mode;
  c.l2norm = (args->flags & KDA_FLAG_L2NORM_QK) != 0;
  c.delta = (args->flags & KDA_FLAG_DELTA_OFF) == 0;
  c.scale = args->scale;
  c.q = args->q;
  c.k = args->k;
  c.v = args->v;
  c.g = args->g;
  c.a = args->a;
  c.A_log = args->A_log;
  c.dt_bias = args->dt_bias;
  c.beta = args->beta;
  c.h0 = args->h0;
  c.o = args->o;
  c.hT = args->hT;
  c.err = args->err;
  c.records = static_cast<unsigned char*>(workspace) + kda::plan_header_bytes(geo.N);
  c.h_chunks = args->h_chunks;
  c.output_pass = output_pass;

  cudaError_t e = cudaSuccess;
  if (geo.cu_seqlens != nullptr) e = kda::launch_plan(c, s);
  if (e == cudaSuccess) {
    if (uses_fused(*args)) {
      e = kda::launch_chunk_fused(c, s);
      // the fused kernel's ring pool is too small for this device's residency
      if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    } else if (output_pass) {
      e = kda::launch_chunk_output_tc(c, s);
    } else {
      e = args->dtype == KDA_DTYPE_BF16 ? kda::launch_chunk_tc(c, s) : kda::launch_chunk_f32(c, s);
    }
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

kda_status kda_chunk_fwd(const kda_chunk_args* args, void* workspace, size_t ws_bytes, kda_stream_t stream) {
  return run_chunk(args, workspace, ws_bytes, stream, false);
}

kda_status kda_chunk_output(const kda_chunk_args* args, void* workspace, size_t ws_bytes, kda_stream_t stream) {
  return run_chunk(args, workspace, ws_bytes, stream, true);
}

namespace {

kda_status check_decode(const kda_decode_args* a, kda::DecodeCall* c) {
  if (a == nullptr) return KDA_ERR_INVALID_ARG;
  if (a->B < 0 || a->H < 1 || a->HV < 1 || a->K < 1 || a->V < 1 || a->num_slots < 0) return KDA_ERR_INVALID_ARG;
  if (a->HV % a->H != 0) return KDA_ERR_INVALID_ARG;
  if (a->flags & ~(KDA_FLAG_L2NORM_QK | KDA_FLAG_CHECK_INDICES)) return KDA_ERR_INVALID_ARG;
  if ((a->flags & KDA_FLAG_CHECK_INDICES) && a->err == nullptr) return KDA_ERR_INVALID_ARG;
  if (!((a->K == 64 || a->K == 128) && (a->V == 64 || a->V == 128))) return KDA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(a->B) * a->HV > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (a->B > 0) {
    if (!a->packed_qkv || !a->a || !a->b || !a->A_log || !a->dt_bias || !a->indices || !a->o)
      return KDA_ERR_INVALID_ARG;
    if (!aligned(a->packed_qkv, 16) || !aligned(a->a, 16) || !aligned(a->b, 2) || !aligned(a->A_log, 4) ||
        !aligned(a->dt_bias, 16) || !aligned(a->indices, 4) || !aligned(a->o, 16))
      return KDA_ERR_INVALID_ARG;
    if (a->num_slots > 0 && (!a->state_pool || !aligned(a->state_pool, 16))) return KDA_ERR_INVALID_ARG;
  }
  if (a->err && !aligned(a->err, 4)) return KDA_ERR_INVALID_ARG;
  c->B = a->B;
  c->H = a->H;
  c->HV = a->HV;
  c->K = a->K;
  c->V = a->V;
  c->num_slots = a->num_slots;
  c->l2norm = (a->flags & KDA_FLAG_L2NORM_QK) != 0;
  c->scale = a->scale;
  c->packed_qkv = a->packed_qkv;
  c->a = a->a;
  c->b = a->b;
  c->A_log = a->A_log;
  c->dt_bias = a->dt_bias;
  c->state_pool = a->state_pool;
  c->indices = a->indices;
  c->o = a->o;
  c->err = a->err;
  c->conv_W = 0;
  c->conv_in = nullptr;
  c->conv_out = nullptr;
  c->conv_w = nullptr;
  c->conv_b = nullptr;
  return KDA_OK;
}

// KDA_FLAG_CHECK_INDICES: the debug check of the slot indices, ahead of the step.
cudaError_t check_indices_if(uint32_t flags, const int32_t* idx, int B, int num_slots, int32_t* err,
                             cudaStream_t s) {
  if (!(flags & KDA_FLAG_CHECK_INDICES)) return cudaSuccess;
  return kda::launch_check_indices(idx, B, num_slots, err, s);
}

}  // namespace

kda_status kda_decode_step(const kda_decode_args* a, kda_stream_t stream) {
  kda::DecodeCall c;
  const kda_status st = check_decode(a, &c);
  if (st != KDA_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = check_indices_if(a->flags, a->indices, a->B, a->num_slots, a->err, s);
  if (e == cudaSuccess) e = kda::launch_decode(c, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode_conv_step(const kda_decode_conv_args* a, kda_stream_t stream) {
  if (a == nullptr) return KDA_ERR_INVALID_ARG;
  kda::DecodeCall c;
  const kda_status st = check_decode(&a->dec, &c);
  if (st != KDA_OK) return st;
  if (a->W < 2 || a->W > 4) return KDA_ERR_UNSUPPORTED;
  if (a->dec.B > 0 && a->dec.num_slots > 0) {
    if (!a->conv_state_in || !a->conv_state_out || !a->conv_weight) return KDA_ERR_INVALID_ARG;
    if (!aligned(a->conv_state_in, 2) || !aligned(a->conv_state_out, 2) || !aligned(a->conv_weight, 4) ||
        (a->conv_bias && !aligned(a->conv_bias, 4)))
      return KDA_ERR_INVALID_ARG;
    if (a->conv_state_in == a->conv_state_out && a->dec.HV != a->dec.H) return KDA_ERR_INVALID_ARG;
  }
  c.conv_W = a->W;
  c.conv_in = a->conv_state_in;
  c.conv_out = a->conv_state_out;
  c.conv_w = a->conv_weight;
  c.conv_b = a->conv_bias;
  // (without slots every row is padding or out of range: the kernel only zeroes o)
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = check_indices_if(a->dec.flags, a->dec.indices, a->dec.B, a->dec.num_slots, a->dec.err, s);
  if (e == cudaSuccess) e = kda::launch_decode(c, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_recurrent_step(const kda_recurrent_args* a, kda_stream_t stream) {
  if (a == nullptr) return KDA_ERR_INVALID_ARG;
  if (a->B < 0 || a->T < 1 || a->H < 1 || a->HV < 1 || a->K < 1 || a->V < 1 || a->num_slots < 0)
    return KDA_ERR_INVALID_ARG;
  if (a->HV % a->H != 0) return KDA_ERR_INVALID_ARG;
  if (a->flags & ~(KDA_FLAG_L2NORM_QK | KDA_FLAG_CHECK_INDICES)) return KDA_ERR_INVALID_ARG;
  if ((a->flags & KDA_FLAG_CHECK_INDICES) && a->err == nullptr) return KDA_ERR_INVALID_ARG;
  if (!((a->K == 64 || a->K == 128) && (a->V == 64 || a->V == 128))) return KDA_ERR_UNSUPPORTED;
  if (a->T > KDA_RECURRENT_MAX_T) return KDA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(a->B) * a->HV > INT32_MAX ||
      static_cast<int64_t>(a->B) * a->T * a->HV * (a->K > a->V ? a->K : a->V) > INT32_MAX)
    return KDA_ERR_INVALID_ARG;
  if (a->B > 0) {
    if (!a->q || !a->k || !a->v || !a->a || !a->b || !a->A_log || !a->dt_bias || !a->indices || !a->o)
      return KDA_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->a, 16) || !aligned(a->b, 2) ||
        !aligned(a->A_log, 4) || !aligned(a->dt_bias, 16) || !aligned(a->indices, 4) || !aligned(a->o, 16))
      return KDA_ERR_INVALID_ARG;
    if (a->num_slots > 0 && (!a->state_pool || !aligned(a->state_pool, 16))) return KDA_ERR_INVALID_ARG;
  }
  if (a->err && !aligned(a->err, 4)) return KDA_ERR_INVALID_ARG;
  kda::RecurrentCall c;
  c.B = a->B;
  c.T = a->T;
  c.H = a->H;
  c.HV = a->HV;
  c.K = a->K;
  c.V = a->V;
  c.num_slots = a->num_slots;
  c.l2norm = (a->flags & KDA_FLAG_L2NORM_QK) != 0;
  c.scale = a->scale;
  c.q = a->q;
  c.k = a->k;
  c.v = a->v;
  c.a = a->a;
  c.b = a->b;
  c.A_log = a->A_log;
  c.dt_bias = a->dt_bias;
  c.state_pool = a->state_pool;
  c.indices = a->indices;
  c.o = a->o;
  c.err = a->err;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = check_indices_if(a->flags, a->indices, a->B, a->num_slots, a->err, s);
  if (e == cudaSuccess) e = kda::launch_recurrent(c, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_head_rmsnorm(const kda_rmsnorm_args* a, kda_stream_t stream) {
  if (a == nullptr || a->R < 0 || !(a->eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (a->V != 64 && a->V != 128) return KDA_ERR_UNSUPPORTED;
  if (a->R > 0) {
    if (!a->x || !a->weight || !a->y) return KDA_ERR_INVALID_ARG;
    if (!aligned(a->x, 16) || !aligned(a->y, 16) || !aligned(a->weight, 16)) return KDA_ERR_INVALID_ARG;
  }
  kda::RmsNormCall c;
  c.R = a->R;
  c.V = a->V;
  c.eps = a->eps;
  c.x = a->x;
  c.weight = a->weight;
  c.y = a->y;
  const cudaError_t e = kda::launch_rmsnorm(c, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

const char* kda_version(void) { return "kda-gb300 0.1.0 sm_103a"; }

kda_status kda_selftest_bounded_wait(int32_t* err, uint64_t limit_ns, kda_stream_t stream) {
  if (err == nullptr || !aligned(err, 4)) return KDA_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > UINT64_C(10000000000)) return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_wait_selftest(err, limit_ns, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_selftest_tcgen05(const kda_tcgen05_probe_args* a, kda_stream_t stream) {
  if (a == nullptr) return KDA_ERR_INVALID_ARG;
  if (a->K != 16 && a->K != 32 && a->K != 64 && a->K != 128) return KDA_ERR_INVALID_ARG;
  if (a->N < 16 || a->N > 256 || a->N % 16 != 0) return KDA_ERR_INVALID_ARG;
  if (a->layout != 0 && a->layout != 1) return KDA_ERR_INVALID_ARG;
  if (a->a_from_tmem != 0 && a->a_from_tmem != 1) return KDA_ERR_INVALID_ARG;
  if (a->reps < 0 || a->reps > 4096) return KDA_ERR_INVALID_ARG;
  if (!a->a || !a->b || !a->d) return KDA_ERR_INVALID_ARG;
  if (!aligned(a->a, 16) || !aligned(a->b, 16) || !aligned(a->d, 16)) return KDA_ERR_INVALID_ARG;
  if (a->cycles && !aligned(a->cycles, 8)) return KDA_ERR_INVALID_ARG;
  if (a->err && !aligned(a->err, 4)) return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_tc05_probe(a->a, a->b, a->d, a->K, a->N, a->layout, a->a_from_tmem, a->reps,
                                               a->cycles, a->err, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
