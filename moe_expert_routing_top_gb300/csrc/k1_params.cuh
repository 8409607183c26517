// k1_params.cuh -- launch parameters of the logits pass of
// moer_topk_signature, shared by its host dispatch and both kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moer {

struct K1Params {
  CUtensorMap tm_logits;  // the logits as a 3-D tiled map (thread-per-row kernel only)
  const float* logits;    // [L][T][E]
  int64_t T;
  int E, k, L;
  uint8_t* ids;          // top-k ids out, or NULL: the caller's [L][T][k], or
  int ids_mask_only;     //   (when set) mask layers only, [m][T][k]
  int32_t* affinity;     // [L][E][E] accumulated, or NULL
  int ntiles;            // token tiles per layer
  int tail_rows;         // tokens in the last tile of a layer (thread-per-row kernel)
  int64_t nitems;        // L * ntiles work items
  uint32_t* status;      // sticky workspace status word
  // 2^24 and 2^8, passed at run time so that the key builder's shift-and-
  // insert stays a multiply-high and a multiply-add (FMA pipe) instead of
  // being folded into a logic op on the integer ALU pipe, which the
  // comparator networks already saturate
  uint32_t key_hi_mul, key_lo_mul;
  // bytes between rows of the co-activation tile, at run time for the same
  // reason: each pair's shared address is then one multiply-add (FMA pipe)
  uint32_t aff_row_bytes;
  // 1 when `affinity` is 8-byte aligned: the fold then adds two neighbouring
  // counts of a row with one 64-bit red (no carry crosses: counts fit in int32)
  int aff_pairs64;
  int16_t slot_of_layer[256];  // mask slot of each layer, -1 if not a mask layer
};

bool tpr_supported(int E, int k);
int tpr_tile_tokens(int E);  // tokens per work item of the thread-per-row kernel
cudaError_t tpr_run(int E, int k, const K1Params& p, int grid, cudaStream_t st);

}  // namespace moer
