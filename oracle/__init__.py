"""CPU oracle for the speculative-decoding verify step (TEST INFRASTRUCTURE).

A plain, slow, fp64 numpy restatement of what the verify step computes,
written from the method's description and independent of the CUDA library:
it shares no code, header, table or helper with it, and neither imports the
other.  Only the test-suite, the smoke check and the bench's CPU-baseline leg
may import it; the product path never does.

Sources (three practitioner pages on speculative decoding):
  * page 1 "投机推理..." (kwkr.cn), §2.1 parallel verify under a causal mask,
    §2.3 / §4.1 the accept rule (accept if p >= q, else with probability p/q),
    §4.3 stop at the first rejection, one consistent resampling source;
  * page 2 "推测解码..." (cf-1.com), §2.1-§2.3 draft/verify flow, the expected
    accepted count (1 - a^(g+1)) / (1 - a), §3.3 KV append and rollback to the
    accepted prefix, §5.4 tree verify with a dynamic rollback path;
  * page 3 "推测解码的工程真相 2026" (blog.lonae.com), formal definition section
    (g drafts + 1 bonus, residual max(0, pi_t - pi_d)) and tree-attention
    section (draft tree of height g and width w verified in one forward).

Modules:
  uniforms       counter-based uniforms (Philox4x64-10 through numpy)
  reject_sample  temperature softmax, accept/reject, residual / bonus sample
  attention      paged-KV append and masked verify attention (batched and
                 token-by-token)
  kv             KV commit: rollback to the accepted prefix, tree-path
                 compaction

Parity status: every function here is pinned by tests under tests/ against
closed forms, exact enumeration, published known-answer vectors or brute
force (see the test module docstrings).
"""
from .uniforms import philox_block, uniforms_for  # noqa: F401
from .reject_sample import (  # noqa: F401
    oracle_reject_sample,
    verify_request,
    UniformChooser,
    inverse_cdf,
    softmax_rows,
    greedy_rows,
    row_law,
    filter_law,
    filter_order,
    FILTER_NEAR,
    NONFINITE,
    INVALID_ARG,
    BAD_TOKEN,
)
from .attention import (  # noqa: F401
    oracle_kv_append,
    oracle_verify_attn,
    oracle_verify_attn_tokenwise,
    gather_positions,
    ancestors_or_self,
)
from .kv import oracle_kv_commit  # noqa: F401
from .lm_head import oracle_lm_head  # noqa: F401
