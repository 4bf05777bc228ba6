// Internal interface between the host entry points (kda_api.cpp) and the
// kernel launchers. Plain structs of device pointers and sizes.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// Where the chunks of a call are. Without cu_seqlens the batch is N sequences
// of T tokens each; with it, chunk_off (in the workspace) holds the first global
// chunk of each sequence, chunk_off[N] the total, chunk_off[N+1] the plan flag
// (1 = cu_seqlens accepted).
struct ChunkGeom {
  int N, T, H;
  int chunks_per_seq;        // ceil(T / 16), uniform batches only
  int max_chunks;            // upper bound of global chunks (grid size of the prep)
  const int32_t* cu_seqlens; // device, or nullptr
  int32_t* chunk_off;        // device, in the workspace (varlen only)
};

// One call of the chunk forward, after host-side validation.
struct ChunkCall {
  ChunkGeom geo;
  int dk, dv;
  int gate_mode, beta_mode;
  bool l2norm, delta;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* a;
  const float* A_log;
  const float* dt_bias;
  const void* beta;
  const float* h0;
  void* o;
  float* hT;
  int32_t* err;
  unsigned char* records;  // workspace after the plan header: per (chunk, head) prep records,
                           // or the fused kernel's pool of global rings
  float* h_chunks;         // per-chunk entering states [chunks, H, dv, dk] (written, or read by the
                           // chunk-parallel output pass), or nullptr
  bool output_pass;        // o from the states in h_chunks instead of the recurrence
};

struct DecodeCall {
  int B, H, HV, K, V, num_slots;
  bool l2norm;
  float scale;
  const void* packed_qkv;
  const void* a;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  const int32_t* indices;
  void* o;
  int32_t* err;
  // causal conv1d + SiLU in front (conv_in == nullptr: packed_qkv is q|k|v already)
  int conv_W;
  const void* conv_in;
  void* conv_out;
  const float* conv_w;
  const float* conv_b;
};

// Workspace layout: [plan header | records]. The header holds N + 2 int32.
inline size_t plan_header_bytes(int N) {
  size_t b = sizeof(int32_t) * static_cast<size_t>(N + 2);
  return (b + 255) & ~static_cast<size_t>(255);
}

struct RecurrentCall {
  int B, T, H, HV, K, V, num_slots;
  bool l2norm;
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
  int32_t* err;
};

struct RmsNormCall {
  long long R;
  int V;
  float eps;
  const void* x;
  const float* weight;
  void* y;
};

// Bytes of one (chunk, head) prep record.
size_t record_bytes_tc(int d);           // bf16 tensor-core path, dk = dv = d
size_t record_bytes_f32(int dk, int dv);  // fp32 path

cudaError_t launch_plan(const ChunkCall& c, cudaStream_t s);
cudaError_t launch_chunk_tc(const ChunkCall& c, cudaStream_t s);
cudaError_t launch_chunk_output_tc(const ChunkCall& c, cudaStream_t s);  // chunk-parallel o from h_chunks
cudaError_t launch_chunk_f32(const ChunkCall& c, cudaStream_t s);
cudaError_t launch_chunk_fused(const ChunkCall& c, cudaStream_t s);  // bf16, dk = dv = 128
size_t fused_workspace_bytes();  // pool of per-cluster global rings (fixed size)
cudaError_t launch_decode(const DecodeCall& c, cudaStream_t s);
cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_check_indices(const int32_t* idx, int B, int num_slots, int32_t* err, cudaStream_t s);
cudaError_t launch_recurrent(const RecurrentCall& c, cudaStream_t s);
cudaError_t launch_recurrent_tc(const RecurrentCall& c, cudaStream_t s);  // T tokens as chunks, tensor cores
cudaError_t launch_recurrent_fma(const RecurrentCall& c, cudaStream_t s);  // T tokens one by one, CUDA cores
cudaError_t launch_rmsnorm(const RmsNormCall& c, cudaStream_t s);
cudaError_t launch_tc05_probe(const void* a, const void* b, float* d, int K, int N, int layout, int a_tmem,
                              int reps, long long* cycles, int32_t* err, cudaStream_t s);

}  // namespace kda
