"""spec_reject_sample_noalloc, the entry point for callers that cannot
allocate device memory (it keeps its scratch in a fixed array inside the
library instead of a caller-provided workspace).

Checked through the C ABI: its outputs equal those of spec_reject_sample on
the same inputs, bit for bit in tokens, paths and lengths and within 1e-5 in
the probe, on two calls in a row (the second reuses the array the first left
behind, with a different shape); sizes beyond the array are refused before
anything is launched.  This file is collected last so that a run stopping at
the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import PROB_ABS, dims_for, tdtype, to_dev  # noqa: E402
from synth import logits_inputs, workload  # noqa: E402


def _inputs(wl, seed):
    lg = logits_inputs(wl, seed=seed)
    dt = tdtype(wl)
    B, M, V = lg["target"].shape
    dev = dict(target=to_dev(lg["target"], dt), draft=to_dev(lg["draft"], dt),
               tokens=to_dev(lg["tokens"], torch.int32),
               parent=None if lg["parent"] is None else to_dev(lg["parent"], torch.int32),
               temperature=to_dev(lg["temperature"], torch.float32))
    return dev, dims_for(wl, B, V=V), (B, M)


def _outputs(B, M):
    return (torch.full((B, M), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, M), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, M, 4), -7.0, dtype=torch.float32, device="cuda"))


def _compare(wl, seed, offset):
    x, dims, (B, M) = _inputs(wl, seed)
    ref = _outputs(B, M)
    ws = sv.workspace(dims)
    sv.spec_reject_sample(x["target"], x["draft"], x["tokens"], x["parent"],
                          x["temperature"], 99, offset, *ref, dims, ws, b_base=3)
    got = _outputs(B, M)
    sv.spec_reject_sample_noalloc(x["target"], x["draft"], x["tokens"], x["parent"],
                                  x["temperature"], 99, offset, *got, dims, b_base=3)
    torch.cuda.synchronize()
    for r, g in zip(ref[:3], got[:3]):
        assert torch.equal(r, g)
    assert torch.max(torch.abs(ref[3] - got[3])).item() <= PROB_ABS
    assert (got[2] >= 0).all()


def test_matches_workspace_entry_point_on_two_calls_in_a_row():
    # first a chain with a 128k vocabulary, then a tree with another shape:
    # the second call runs on whatever the first left in the shared array
    _compare(workload("chain_gqa_128k"), seed=21, offset=0)
    _compare(workload("tree_64").scaled(B=4), seed=22, offset=1)


def test_same_inputs_twice():
    wl = workload("chain_7b")
    _compare(wl, seed=23, offset=5)
    _compare(wl, seed=23, offset=5)


def test_refuses_sizes_beyond_its_scratch():
    # 16384 requests x 5 rows of a 16-logit vocabulary: the kernels these
    # sizes run on (the staged ones) need 16 MB of scratch, far beyond the
    # 1 MiB array.  The
    # buffers have the full sizes, so nothing could be read out of bounds
    # even if the call went ahead.
    B, M, V = 16384, 5, 16
    dims = sv.make_dims(B=B, M=M, V=V)
    t = torch.zeros(B, M, V, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(B, M, dtype=torch.int32, device="cuda")
    f = torch.ones(B, dtype=torch.float32, device="cuda")
    a = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_reject_sample_noalloc(t, t, i, None, f, 1, 0, i, i.clone(), a, None, dims)
    assert e.value.code == 3
    # the one-kernel path's scratch: 40000 requests' chunk statistics, row
    # normalisers and counters (over 6 MB)
    B = 40000
    dims = sv.make_dims(B=B, M=M, V=64, reject_impl=sv.REJECT_FUSED)
    t = torch.zeros(B, M, 64, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(B, M, dtype=torch.int32, device="cuda")
    f = torch.ones(B, dtype=torch.float32, device="cuda")
    a = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_reject_sample_noalloc(t, t, i, None, f, 1, 0, i, i.clone(), a, None, dims)
    assert e.value.code == 3
