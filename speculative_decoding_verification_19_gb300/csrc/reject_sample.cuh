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

constexpr int kRsMaxM = kMaxNodes;

// Law at the node where a request draws: row maxima and normalisers of the
// node's target / draft rows, and the masses of the residuals taken so far.
struct DecideCtx {
  float mT, mD;          // row maxima of the node's target / draft rows
  float invST, invSD;    // 1 / row sums (fp32); 1 / kept mass for a filtered row
  float cs;              // log2(e) / T
  int nrej;              // rejections so far at this node (working P = P_nrej)
  // filtered laws (top-k / top-p): a token of the target (draft) row is kept
  // iff its logit is above vT (vD), or equal with an index at most iT (iD);
  // -inf and INT_MAX keep every token
  float vT, vD;
  int iT, iD;
  float invZ[kRsMaxM];   // 1 / Z_j of the residuals taken so far (element path)
  double Z[kRsMaxM];     // Z_j in fp64 (accept-test path)
};

// A draw left for the residual kernels: the law, the node, the number of
// accepted drafts and the uniform.
struct DrawState {
  DecideCtx c;
  double u;
  int node, a, pending, pad;
};

// The kept prefix of a filtered row (see DecideCtx) and its mass
// K = sum over kept tokens of exp2((z - m) cs); K = 0: the row is not
// filtered.
struct FilterInfo {
  float v;
  int idx;
  double K;
};

struct RsArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* parent;
  const float* temperature;
  const int32_t* top_k;  // [B] or NULL
  const float* top_p;    // [B] or NULL
  uint64_t seed, offset, b_base;
  int32_t* out_tokens;
  int32_t* path;
  int32_t* accepted_len;
  float* probe;
  spec_dims d;
  void* ws;
  bool stats_ready = false;  // the chunk statistics are already in the workspace
};

int rs_chunk_elems(int logits_dtype);       // statistics chunk (one warp task)
int rs_max_vocab(int logits_dtype);
// rs_launch picks the kernels (spec_dims.reject_impl): the fused one-kernel
// path (reject_fused.cu) when the shape allows it, else the staged four.
// Returns cudaErrorNotSupported when the fused path is asked for and the
// shape does not allow it.
cudaError_t rs_launch(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches);
// The one-kernel path (statistics, decisions and draws in one launch) takes
// chains with 16-byte aligned rows.
bool rso_supported(const spec_dims& d, bool aligned, bool chain);
// Lays out the one-kernel path's scratch from byte offset `off` (256-byte
// aligned) and returns the end.
size_t rsf_layout(const spec_dims& d, size_t off, WsLayout* L);
// The tree walk by clusters (rs_tree_walk.cu): trees of 16-byte aligned
// rows without filters.  inputs_ready: launched right after the statistics
// kernel (which lets it start once everything before that kernel has
// completed); false after the LM heads (it waits for its predecessor).
bool rs_tree_walk_supported(const spec_dims& d, bool aligned, bool tree, bool filters);
cudaError_t rs_tree_walk_launch(const RsArgs& a, const WsLayout& lay, bool inputs_ready,
                                cudaStream_t st);

}  // namespace specv
