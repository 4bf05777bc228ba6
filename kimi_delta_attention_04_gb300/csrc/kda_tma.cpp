// Host-side encoding of the fused kernel's TMA descriptors. The driver entry
// point is looked up through the runtime, so the library needs no libcuda link.
#include "kda_tma.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace kda {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, size_t elem, int D, int H, long long tokens) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem, static_cast<cuuint64_t>(H) * D * elem};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1u, 16u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t encode_input_maps(const ChunkCall& c, TmaInputMaps* m) {
  const long long tokens = c.geo.cu_seqlens ? static_cast<long long>(c.geo.T)
                                            : static_cast<long long>(c.geo.N) * c.geo.T;
  if (tokens == 0) return cudaSuccess;
  const int H = c.geo.H, D = c.dk;
  bool ok = encode3d(&m->q, c.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, H, tokens) &&
            encode3d(&m->k, c.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, H, tokens) &&
            encode3d(&m->v, c.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, H, tokens);
  if (ok && (c.gate_mode == 1 || c.gate_mode == 2))  // per-channel gate tiles (not the per-head one)
    ok = encode3d(&m->a, c.gate_mode == 1 ? static_cast<const void*>(c.g) : static_cast<const void*>(c.a),
                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, H, tokens);
  return ok ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace kda
