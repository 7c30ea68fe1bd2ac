"""GPU parity of spec_verify_attn at the benchmarked sizes.

The bench times whole batches: 32 requests of the 128k-vocabulary chain
workload, 16 trees of 64 nodes, 128 requests of the stress workload (contexts
of 4k to 32k tokens, a 10 GB cache).  At those sizes each CTA range of the
persistent tensor-core kernel crosses many (request, KV head) segments and
split pairs, and the merge runs under a plan of a thousand segments or more;
the smaller parity cases do not reach that.  So the call here is the bench's
own call (same dims, same automatic kernel choice, the cache drawn on the
device), and a spread of its requests -- the shortest and longest context,
the first and the last request and four chosen at random -- is compared
element by element with the fp64 oracle run on those requests alone (their
pages read back before the call): outputs within 2e-2 absolute + 1e-2
relative, log-sum-exp within 1e-3, and the appended rows of each sampled
request bit-exact.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import assert_attn_close  # noqa: E402
from oracle import oracle_verify_attn  # noqa: E402
from synth import kv_inputs_device, logits_inputs, workload  # noqa: E402


def _sample(ctx, seed):
    B = len(ctx)
    pick = {int(np.argmin(ctx)), int(np.argmax(ctx)), 0, B - 1}
    rng = np.random.default_rng(seed)
    while len(pick) < min(B, 8):
        pick.add(int(rng.integers(B)))
    return sorted(pick)


def _pages(kv, b):
    bt = kv["block_table"][b]
    pages = bt[bt >= 0].astype(np.int64)
    idx = torch.from_numpy(pages).to(kv["k_cache"].device)
    kc = kv["k_cache"].index_select(0, idx).float().cpu().numpy()
    vc = kv["v_cache"].index_select(0, idx).float().cpu().numpy()
    return kc, vc, len(pages)


@pytest.mark.parametrize("name,seed", [("chain_gqa_128k", 0), ("chain_gqa_128k", 2),
                                       ("tree_64", 0), ("stress_gqa_152k", 0)])
def test_bench_batch_against_oracle(name, seed):
    wl = workload(name)
    dev = torch.device("cuda")
    kv = kv_inputs_device(wl, seed, dev)
    parent = None
    if wl.is_tree:
        parent = logits_inputs(wl.scaled(V=16), seed)["parent"]
    B = wl.B
    ctx = kv["ctx_lens"]
    reqs = _sample(ctx, seed + 100)
    before = {b: _pages(kv, b) for b in reqs}
    dt = torch.bfloat16
    dims = sv.make_dims(B=B, M=wl.M, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D,
                        max_blocks=kv["max_blocks"], num_blocks=kv["num_blocks"],
                        V=wl.V, kv_dtype=dt, logits_dtype=dt)
    ws = sv.workspace(dims)
    bt = torch.from_numpy(kv["block_table"]).to(dev)
    cl = torch.from_numpy(ctx).to(dev)
    par = None if parent is None else torch.from_numpy(parent).to(dev)
    out = torch.full_like(kv["q"], float("nan"))
    lse = torch.full(kv["q"].shape[:3], float("nan"), dtype=torch.float32, device=dev)
    sv.spec_verify_attn(kv["q"], kv["k_new"], kv["v_new"], kv["k_cache"], kv["v_cache"],
                        bt, cl, par, out, lse, dims, ws)
    torch.cuda.synchronize()
    assert sv.device_status(ws) == 0
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    for b in reqs:
        kc, vc, npg = before[b]
        table = np.arange(npg, dtype=np.int32)[None]
        o_out, o_lse, o_kc, o_vc = oracle_verify_attn(
            kv["q"][b:b + 1].float().cpu().numpy(), kc, vc, table, ctx[b:b + 1],
            kv["k_new"][b:b + 1].float().cpu().numpy(),
            kv["v_new"][b:b + 1].float().cpu().numpy(),
            parent=None if parent is None else parent[b:b + 1], block=wl.block)
        assert_attn_close(out[b:b + 1].float().cpu().numpy(), o_out,
                          lse[b:b + 1].cpu().numpy(), o_lse)
        g_kc, g_vc, _ = _pages(kv, b)
        assert np.array_equal(g_kc, o_kc.astype(np.float32)), b
        assert np.array_equal(g_vc, o_vc.astype(np.float32)), b
