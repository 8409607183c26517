// k1_params.cuh -- launch parameters shared by the host dispatch of
// moer_topk_signature and the thread-per-row kernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moer {

// Thread-per-row kernel: one (layer, 32-token tile) work item per tile.
struct TprParams {
  const float* logits;
  int64_t T;
  int k, L, m;
  uint8_t* topk;
  uint8_t* blk_cnt;
  int32_t* affinity;
  const int32_t* tok_blk;
  int ntiles;
  int64_t nitems;
  uint32_t* status;
  uint32_t* call_flag;
  int16_t slot_of_layer[256];
};

bool tpr_supported(int E, int k);
cudaError_t tpr_run(int E, int k, const TprParams& p, int grid, cudaStream_t st);

}  // namespace moer
