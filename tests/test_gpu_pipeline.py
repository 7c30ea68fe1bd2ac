"""GPU parity of consecutive verify steps through the whole public API.

Each step runs append + attention, reject-sample and commit, and the next
step's attention reads the context lengths that the previous commit wrote.
Every kernel of that chain is a programmatic dependent launch of the one
before it, so this covers the ordering of reads and writes across calls.

A host pipeline of the oracle runs beside it on its own cache and lengths.
At every step these must match:
- the attention output (within the stated tolerance);
- the decisions (bit-exact; the seeds are chosen with no draw near a
  threshold);
- the committed cache (bit-exact outside the freed slots);
- the new lengths (bit-exact).
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import (NEAR, assert_attn_close, cache_equal_except, dims_for,  # noqa: E402
                     tdtype, to_dev)
from oracle import oracle_kv_commit, oracle_reject_sample, oracle_verify_attn  # noqa: E402
from synth import kv_inputs_host, logits_inputs, workload  # noqa: E402


def _run_steps(wl, ctx0, steps, impl, parent_seed=None):
    B, M = len(ctx0), wl.M
    dt = tdtype(wl)
    # a block table with room for every step's new rows
    kv = kv_inputs_host(wl, seed=31, B=B, ctx=ctx0 + steps * M)
    dims = dims_for(wl, B, kv["max_blocks"], kv["num_blocks"], impl=impl)
    ws = sv.workspace(dims)
    kc, vc = to_dev(kv["k_cache"], dt), to_dev(kv["v_cache"], dt)
    bt = to_dev(kv["block_table"], torch.int32)
    lens = [to_dev(ctx0.astype(np.int32), torch.int32),
            torch.full((B,), -7, dtype=torch.int32, device="cuda")]
    o_kc, o_vc = kv["k_cache"].copy(), kv["v_cache"].copy()
    o_ctx = ctx0.astype(np.int32).copy()
    for s in range(steps):
        new = kv_inputs_host(wl, seed=200 + s, B=B, ctx=np.zeros(B, dtype=np.int32))
        lg = logits_inputs(wl, seed=300 + s, B=B)
        cur, nxt = lens[s % 2], lens[(s + 1) % 2]
        q, kn, vn = (to_dev(new[k], dt) for k in ("q", "k_new", "v_new"))
        par = None if lg["parent"] is None else to_dev(lg["parent"], torch.int32)
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        toks = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
        path = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
        acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        # the whole step is enqueued before anything is read back
        sv.spec_verify_attn(q, kn, vn, kc, vc, bt, cur, par, out, lse, dims, ws)
        sv.spec_reject_sample(to_dev(lg["target"], dt), to_dev(lg["draft"], dt),
                              to_dev(lg["tokens"], torch.int32), par,
                              to_dev(lg["temperature"], torch.float32), 77, s, toks, path,
                              acc, None, dims, ws)
        sv.kv_commit(kc, vc, bt, cur, nxt, path, acc, dims, ws)
        torch.cuda.synchronize()
        assert sv.device_status(ws) == 0

        o_out, o_lse, o_kc, o_vc = oracle_verify_attn(
            new["q"], o_kc, o_vc, kv["block_table"], o_ctx, new["k_new"], new["v_new"],
            parent=lg["parent"], block=wl.block)
        o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], lg["parent"],
                                 lg["temperature"], 77, s)
        assert np.all(o["margin"] >= NEAR), "seed with a near-threshold draw"
        hi = o_ctx + M
        o_kc, o_vc, o_ctx = oracle_kv_commit(o_kc, o_vc, kv["block_table"], o_ctx, o["path"],
                                             o["accepted_len"], block=wl.block)

        assert_attn_close(out.float().cpu().numpy(), o_out, lse.cpu().numpy(), o_lse)
        assert np.array_equal(acc.cpu().numpy(), o["accepted_len"]), s
        assert np.array_equal(path.cpu().numpy(), o["path"]), s
        assert np.array_equal(toks.cpu().numpy(), o["out_tokens"]), s
        assert np.array_equal(nxt.cpu().numpy(), o_ctx), s
        for g, oc in ((kc, o_kc), (vc, o_vc)):
            assert cache_equal_except(g.float().cpu().numpy(), oc.astype(np.float32),
                                      kv["block_table"], o_ctx, hi), s


@pytest.mark.parametrize("impl", [sv.ATTN_TENSOR_CORES, sv.ATTN_CUDA_CORES])
def test_chain_steps(impl):
    wl = workload("chain_gqa_128k").scaled(gamma=3, V=2048)
    _run_steps(wl, np.array([0, 17, 300, 1500, 64]), steps=3, impl=impl)


def test_tree_steps():
    wl = workload("tree_64").scaled(Hq=4, Hkv=2, V=2048)
    _run_steps(wl, np.array([5, 700, 40]), steps=3, impl=sv.ATTN_TENSOR_CORES)
