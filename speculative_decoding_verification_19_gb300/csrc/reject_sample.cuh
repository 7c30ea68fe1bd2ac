// Internal interface between the C ABI layer and the reject-sample kernels.
#pragma once

#include "common.cuh"

namespace specv {

// Statistics of one chunk of a logits row: the chunk maximum m and
// s = sum over the chunk of exp2((z - m) * log2(e) / T).
struct RowStat {
  float m;
  float pad;
  double s;
};

struct RsArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* parent;
  const float* temperature;
  uint64_t seed, offset, b_base;
  int32_t* out_tokens;
  int32_t* path;
  int32_t* accepted_len;
  float* probe;
  spec_dims d;
  void* ws;
};

int rs_chunk_elems(int logits_dtype);
int rs_max_vocab(int logits_dtype);
cudaError_t rs_launch(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);

}  // namespace specv
