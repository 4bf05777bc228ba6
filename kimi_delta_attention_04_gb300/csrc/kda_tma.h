// Tensor maps (TMA descriptors) for the per-chunk input tiles of the fused
// chunk kernel: one 3-D map [tokens][heads][channels] per input, box
// 16 tokens x 1 head x 128 channels, rows past the end read as zero.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

struct TmaInputMaps {
  CUtensorMap q, k, v, a;  // a: gate inputs or log-decay g (fp32); unused without a gate
};

// Host: fills the maps for a bf16 dk = dv = 128 call. Returns cudaErrorInvalidValue
// if the driver cannot encode them.
cudaError_t encode_input_maps(const ChunkCall& c, TmaInputMaps* m);

}  // namespace kda
