// Internal interface of the LM-head GEMM with the reject-sample statistics
// in its epilogue (lm_head.cu).
#pragma once

#include "common.cuh"
#include "reject_sample.cuh"

namespace specv {

// H a multiple of 64, V a multiple of 256 (bf16 rows, 16-byte aligned).
bool lm_head_supported(int R, int H, int V);

// logits[R, V] = hidden[R, H] weight[V, H]^T (bf16, fp32 accumulation).
// With stats != nullptr also each row's chunk statistics (2048-logit
// chunks, the layout the reject-sample kernels read: row r is node r % M
// of request r / M, `which` = 0 target / 1 draft) at the temperature of its
// request.  Launches one kernel.
cudaError_t lm_head_launch(const void* hidden, const void* weight, int R, int H, int V,
                           void* logits, RowStat* stats, int which, int M, int n_chunks,
                           const float* temperature, const spec_dims& d, uint32_t* status,
                           cudaStream_t st, int* launches);

}  // namespace specv
