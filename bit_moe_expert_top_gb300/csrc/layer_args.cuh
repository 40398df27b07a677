// The single-launch 2-bit decode layer (gemv_lut.cu): the arguments beyond
// the fused FC1 + FC2 launch's (routing and grouping outputs, the combine's
// output) and its launch.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace moe {

struct LayerArgs {
  const float* logits;
  int T, E, k;
  int32_t* ids;
  float* w;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  void* y;
  void* out;
  int out_fmt;
};
bool layer_supported(int T, int E, int k);
cudaError_t launch_w2_decode_layer(const LayerArgs& la, const MMArgs& fc1, const MMArgs& fc2, void* ws,
                                   cudaStream_t s);

}  // namespace moe
