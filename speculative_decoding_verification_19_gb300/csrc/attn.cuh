// Internal interface between the C ABI layer and the attention kernels.
#pragma once

#include "common.cuh"

namespace specv {

struct AttnArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* parent;
  void* out;
  float* lse;
  spec_dims d;
  float scale;
  void* ws;
};

size_t attn_simt_smem_bytes(int R, int D);
cudaError_t attn_launch_simt(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);

}  // namespace specv
