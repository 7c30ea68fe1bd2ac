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

// CTAs of the persistent tensor-core kernel never exceed this (partials are
// sized for it).
constexpr int kMaxAttnCtas = 512;

// Floats per partial row of the tensor-core path: D outputs, the log2-sum-exp
// at index D, padded so every row starts on a 16-byte boundary.
__host__ __device__ constexpr int tc_part_stride(int D) { return D + 4; }

size_t attn_simt_smem_bytes(int R, int D);
size_t attn_tc_part_floats(const spec_dims& d);
cudaError_t kv_append_launch(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);
cudaError_t attn_launch_simt(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);
cudaError_t attn_launch_tc(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);

}  // namespace specv
