// Internal interface of the LM-head GEMM with the reject-sample statistics
// in its epilogue (lm_head.cu).
#pragma once

#include "common.cuh"
#include "reject_sample.cuh"

namespace specv {

// H a multiple of 64, V a multiple of 256 (bf16 rows, 16-byte aligned).
bool lm_head_supported(int R, int H, int V);

// Work units of the kernel (128-row tiles x 2048-column chunks).  A call
// with statistics may split each unit into up to kLmMaxPieces pieces when
// the workspace holds their partial statistics: [2][units][kLmMaxPieces]
// [128] RowStat and [2][units][4] u32 counters (zero between calls), laid
// out only for up to kLmSplitMaxUnits units (beyond that the waves of whole
// units are already full to within a ninth).
constexpr int kLmMaxPieces = 4;
constexpr int64_t kLmSplitMaxUnits = 1216;
int64_t lm_head_units(int R, int V);

// logits[R, V] = hidden[R, H] weight[V, H]^T (bf16, fp32 accumulation).
// With stats != nullptr also each row's chunk statistics (2048-logit
// chunks, the layout the reject-sample kernels read: row r is node r % M
// of request r / M, `which` = 0 target / 1 draft) at the temperature of its
// request; part / cnt: the split statistics' workspace (nullptr: units are
// not split).  Launches one kernel.
cudaError_t lm_head_launch(const void* hidden, const void* weight, int R, int H, int V,
                           void* logits, RowStat* stats, int which, int M, int n_chunks,
                           const float* temperature, const spec_dims& d, uint32_t* status,
                           RowStat* part, uint32_t* cnt, cudaStream_t st, int* launches);

}  // namespace specv
