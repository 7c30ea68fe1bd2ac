"""Bounded device waits that run out, on purpose, without faulting or hanging.

Every spin-wait of the kernels gives up after spec_dims.wait_limit_kcycles
thousand SM clocks and raises SPEC_ERR_TIMEOUT; work the CTA already issued
(copies into its shared memory, MMAs into its tensor memory) is still
waited for before it exits.  These tests set a limit of a thousand clocks,
far below what a wait takes when it has real work behind it, and check that

* the call returns and the status word carries SPEC_ERR_TIMEOUT;
* reject-sample reports every request as failed (accepted_len = -1), not
  decisions made on statistics a gave-up wait left unwritten;
* an ordinary call right after, in the same process, on a re-initialised
  workspace, matches the oracle again.

Nothing here faults, traps or waits without a limit: the kernels' waits are
all bounded, and the short limit only makes them give up sooner.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import (assert_attn_close, compare_reject, dims_for, gpu_attn,  # noqa: E402
                     gpu_reject, oracle_attn, tdtype, to_dev)
from oracle import oracle_reject_sample  # noqa: E402
from synth import kv_inputs_host, logits_inputs, workload  # noqa: E402

TIMEOUT_BIT = 1 << 7
TINY = 1  # thousand SM clocks


def _flush_l2():
    """Evict the inputs from L2 (a write larger than it), so that the first
    bulk copies come from HBM and outlast the thousand-clock limit."""
    buf = torch.empty(96 << 20, dtype=torch.float32, device="cuda")
    buf.fill_(1.0)
    torch.cuda.synchronize()


def test_attention_wait_gives_up_then_recovers():
    # one 40k-token request: each (request, KV head) pair is split over
    # about twenty CTAs, so the CTA holding a pair's first tile waits for the
    # others' partials, and the copy pipeline waits for its loads
    wl = workload("chain_gqa_128k")
    kv = kv_inputs_host(wl, seed=31, B=1, ctx=np.array([40000]))
    B = 1
    dims = dims_for(wl, B, kv["max_blocks"], kv["num_blocks"], impl=sv.ATTN_TENSOR_CORES)
    dims.wait_limit_kcycles = TINY
    ws = sv.workspace(dims)
    g = gpu_attn(wl, kv, dims=dims, ws=ws)
    assert g["status"] & TIMEOUT_BIT
    # the same shape with the default limit, on a re-initialised workspace
    dims.wait_limit_kcycles = 0
    ws = sv.workspace(dims)
    g = gpu_attn(wl, kv, dims=dims, ws=ws)
    assert g["status"] == 0
    o_out, o_lse, o_kc, _ = oracle_attn(wl, kv)
    assert_attn_close(g["out"], o_out, g["lse"], o_lse)


@pytest.mark.parametrize("impl", [sv.REJECT_STAGED, sv.REJECT_FUSED])
def test_reject_wait_gives_up_then_recovers(impl):
    # the full stress batch: 350 MB of logits, so that the statistics'
    # copies queue at HBM and some wait outlasts the thousand-clock limit
    wl = workload("stress_gqa_152k")
    lg = logits_inputs(wl, seed=32)
    B, M, V = lg["target"].shape
    dims = dims_for(wl, B, V=V)
    dims.reject_impl = impl
    dims.wait_limit_kcycles = TINY
    ws = sv.workspace(dims)
    _flush_l2()
    g = gpu_reject(wl, lg, seed=5, offset=0, dims=dims, ws=ws)
    assert g["status"] & TIMEOUT_BIT
    # no request is decided on lost statistics: both paths fail every
    # request of the call
    a = g["accepted_len"]
    assert np.all(a == -1)
    dims.wait_limit_kcycles = 0
    ws = sv.workspace(dims)
    g = gpu_reject(wl, lg, seed=5, offset=1, dims=dims, ws=ws)
    assert g["status"] == 0
    o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], lg["parent"],
                             lg["temperature"], 5, 1)
    compare_reject(g, o)


def test_tree_walk_wait_gives_up_then_recovers():
    # trees of aligned rows: the statistics stream and the cluster walk,
    # whose exchanges wait (bounded) on mbarriers that the other CTAs of the
    # cluster arrive on; after a wait gives up the walk still meets the
    # cluster barrier at its end, and every request of the call fails
    # rows of the stress vocabulary: 623 MB of logits, more than L2 holds even
    # right after they are written, so the statistics' copies come from HBM
    wl = workload("tree_64").scaled(B=16, V=152064)
    lg = logits_inputs(wl, seed=34)
    B, M, V = lg["target"].shape
    dims = dims_for(wl, B, V=V)
    dims.wait_limit_kcycles = TINY
    ws = sv.workspace(dims)
    _flush_l2()
    g = gpu_reject(wl, lg, seed=6, offset=0, dims=dims, ws=ws)
    assert g["status"] & TIMEOUT_BIT
    assert np.all(g["accepted_len"] == -1)
    dims.wait_limit_kcycles = 0
    ws = sv.workspace(dims)
    g = gpu_reject(wl, lg, seed=6, offset=1, dims=dims, ws=ws)
    assert g["status"] == 0
    o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], lg["parent"],
                             lg["temperature"], 6, 1)
    compare_reject(g, o)


def test_noalloc_wait_gives_up_then_recovers():
    # the no-allocation entry point cannot report its status word: a wait
    # that gave up shows as accepted_len = -1 for the requests it touched
    wl = workload("stress_gqa_152k").scaled(B=48)  # its scratch fits the 1 MiB array
    lg = logits_inputs(wl, seed=33)
    B, M, V = lg["target"].shape
    dims = dims_for(wl, B, V=V)
    dims.wait_limit_kcycles = TINY
    dt = tdtype(wl)
    args = [to_dev(lg["target"], dt), to_dev(lg["draft"], dt), to_dev(lg["tokens"], torch.int32),
            None, to_dev(lg["temperature"], torch.float32), 9, 0]
    out = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    _flush_l2()
    sv.spec_reject_sample_noalloc(*args, out, path, acc, None, dims)
    torch.cuda.synchronize()
    a = acc.cpu().numpy()
    assert np.all((a == -1) | (a >= 0))
    timed_out = a == -1
    dims.wait_limit_kcycles = 0
    sv.spec_reject_sample_noalloc(*args, out, path, acc, None, dims)
    torch.cuda.synchronize()
    o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], None,
                             lg["temperature"], 9, 0)
    g = dict(out_tokens=out.cpu().numpy(), path=path.cpu().numpy(),
             accepted_len=acc.cpu().numpy(), status=0)
    compare_reject(g, o)
    # with a thousand-clock limit the statistics stream cannot finish
    assert timed_out.any()
