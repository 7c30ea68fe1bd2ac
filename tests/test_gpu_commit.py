"""GPU parity of kv_commit: the whole cache bit-exact against the oracle
except the freed slots [new_ctx, ctx+M), and the new context lengths."""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import cache_equal_except, dims_for, tdtype, to_dev  # noqa: E402
from oracle import oracle_kv_commit, oracle_reject_sample  # noqa: E402
from synth import kv_inputs_host, logits_inputs, workload  # noqa: E402


def _commit(wl, kv, path, acc, alias=False):
    dt = tdtype(wl)
    B = kv["block_table"].shape[0]
    dims = dims_for(wl, B, kv["max_blocks"], kv["num_blocks"])
    ws = sv.workspace(dims)
    kc = to_dev(kv["k_cache"], dt)
    vc = to_dev(kv["v_cache"], dt)
    bt = to_dev(kv["block_table"], torch.int32)
    ctx = to_dev(kv["ctx_lens"], torch.int32)
    new = ctx if alias else torch.empty_like(ctx)
    sv.kv_commit(kc, vc, bt, ctx, new, to_dev(path, torch.int32),
                 to_dev(acc, torch.int32), dims, ws)
    torch.cuda.synchronize()
    return (kc.float().cpu().numpy(), vc.float().cpu().numpy(),
            new.cpu().numpy(), sv.device_status(ws))


@pytest.mark.parametrize("name,alias", [("tree_64", False), ("tree_64", True),
                                        ("tree_wide_128", False)])
def test_tree_compaction(name, alias):
    wl = workload(name).scaled(V=2000)
    B = 6
    lg = logits_inputs(wl, seed=8, B=B)
    kv = kv_inputs_host(wl.scaled(Hq=4, Hkv=4), seed=8, B=B,
                        ctx=np.array([0, 15, 16, 100, 4000, 33]))
    o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"],
                             lg["parent"], lg["temperature"], 5, 0)
    assert o["accepted_len"].max() >= 2          # some paths move slots
    wlk = wl.scaled(Hq=4, Hkv=4)
    gk, gv, gn, st = _commit(wlk, kv, o["path"], o["accepted_len"], alias)
    ok, ov, on = oracle_kv_commit(kv["k_cache"], kv["v_cache"], kv["block_table"],
                                  kv["ctx_lens"], o["path"], o["accepted_len"])
    assert st == 0
    assert np.array_equal(gn, on)
    hi = kv["ctx_lens"] + wl.M
    assert cache_equal_except(gk, ok.astype(np.float32), kv["block_table"], on, hi)
    assert cache_equal_except(gv, ov.astype(np.float32), kv["block_table"], on, hi)


def test_chain_is_length_update_and_failed_requests():
    wl = workload("chain_gqa_128k")
    B = 4
    kv = kv_inputs_host(wl.scaled(Hq=8, Hkv=2), seed=9, B=B,
                        ctx=np.array([10, 200, 3000, 17]))
    path = np.tile(np.arange(wl.M, dtype=np.int32), (B, 1))
    acc = np.array([0, 8, -1, 3], dtype=np.int32)
    path[2] = -1
    gk, gv, gn, st = _commit(wl.scaled(Hq=8, Hkv=2), kv, path, acc)
    assert st == 0
    assert gn.tolist() == [11, 209, 3000, 21]
    assert np.array_equal(gk, kv["k_cache"]) and np.array_equal(gv, kv["v_cache"])


def test_bad_path_is_rejected():
    wl = workload("tree_64").scaled(Hq=2, Hkv=2)
    kv = kv_inputs_host(wl, seed=10, B=2, ctx=np.array([5, 9]))
    path = np.full((2, wl.M), -1, dtype=np.int32)
    path[:, 0] = 0
    path[0, 1] = 0            # path[1] must be >= 1
    path[1, 1] = 3
    acc = np.array([1, 1], dtype=np.int32)
    gk, gv, gn, st = _commit(wl, kv, path, acc)
    assert st == (1 << 1)
    assert gn.tolist() == [5, 11]
