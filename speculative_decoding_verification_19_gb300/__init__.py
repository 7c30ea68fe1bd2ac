"""GB300-native verify step of speculative decoding.

The compute lives in libspecverify.so (hand-written CUDA for sm_103a, C ABI
in include/spec_verify.h).  This package is its thin Python binding:

  spec_verify_attn    KV append + masked verify attention over a paged cache
  spec_reject_sample  temperature softmax, accept/reject, residual/bonus draw
                      (greedy at temperature 0; top-k / top-p restricted laws)
  spec_lm_head        LM-head logits on the tensor cores
  spec_reject_sample_lm_head  LM heads + decisions, statistics in the epilogue
  kv_commit           rollback / tree-path compaction of the KV cache

plus helpers to size and initialise the caller-owned workspace and to read
the device status word.
"""
from ._native import (  # noqa: F401
    ATTN_AUTO,
    ATTN_CUDA_CORES,
    ATTN_TENSOR_CORES,
    REJECT_AUTO,
    REJECT_FUSED,
    REJECT_STAGED,
    EXPORTS,
    LIB_PATH,
    SPEC_BF16,
    SPEC_F32,
    SpecDims,
    SpecError,
    device_status,
    dtype_code,
    kv_commit,
    lib,
    make_dims,
    philox_block,
    spec_lm_head,
    spec_reject_sample,
    spec_reject_sample_lm_head,
    spec_reject_sample_noalloc,
    spec_verify_attn,
    workspace,
    workspace_size,
)
