// Internal interface between the C ABI layer and the commit kernel.
#pragma once

#include "common.cuh"

namespace specv {

struct CommitArgs {
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  int32_t* new_ctx_lens;
  const int32_t* path;
  const int32_t* accepted_len;
  spec_dims d;
  void* ws;
};

cudaError_t commit_launch(const CommitArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);

}  // namespace specv
