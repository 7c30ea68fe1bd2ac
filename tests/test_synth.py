"""Checks of the seeded input generators (shapes, tree structure, draws)."""
import numpy as np
import torch
from scipy import stats

from synth import (WORKLOADS, bf16_round, kv_layout, logits_inputs,
                   random_tree, workload)


def test_bf16_round_matches_torch():
    x = np.random.default_rng(0).normal(0, 3, 100_000).astype(np.float32)
    x[:4] = [np.inf, -np.inf, 0.0, -0.0]
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(bf16_round(x), ref)


def test_random_tree_is_bfs_and_ancestor_closed():
    rng = np.random.default_rng(1)
    for _ in range(50):
        par = random_tree(rng, 4, 4, 64)
        assert par[0] == -1 and np.all(par[1:] >= 0)
        assert np.all(par[1:] < np.arange(1, 64))
        depth = np.zeros(64, dtype=int)
        for n in range(1, 64):
            depth[n] = depth[par[n]] + 1
        assert depth.max() <= 4
        assert np.all(np.diff(depth) >= 0)                # BFS order
        assert max(np.bincount(par[1:], minlength=64)) <= 4


def test_full_tree_size():
    par = random_tree(np.random.default_rng(2), 4, 4, 341)
    assert len(par) == 341 and np.bincount(par[1:]).max() == 4


def test_workload_shapes():
    wl = workload("tiny_chain")
    d = logits_inputs(wl, 0)
    assert d["target"].shape == (1, 5, 32) and d["parent"] is None
    assert d["tokens"].shape == (1, 5)
    t = workload("tree_64").scaled(V=64)
    d = logits_inputs(t, 0, B=2)
    assert d["parent"].shape == (2, 64)
    w = workload("tree_wide_128").scaled(V=64)
    d = logits_inputs(w, 0, B=2)
    par = d["parent"]
    assert par.shape == (2, 128) and np.all(par[:, 0] == -1)
    assert np.all(par[:, 1:] < np.arange(1, 128)) and np.all(par[:, 1:] >= 0)
    assert max(np.bincount(p[1:]).max() for p in par) <= 8
    assert w.B * w.tree_width <= 256
    lay = kv_layout(WORKLOADS["chain_gqa_128k"], 0)
    need = (lay["ctx_lens"] + 9 + 15) // 16
    assert np.all((lay["block_table"] >= 0).sum(1) == need)
    used = lay["block_table"][lay["block_table"] >= 0]
    assert len(np.unique(used)) == used.size           # no block shared


def test_draft_tokens_follow_q():
    # Gumbel-max draws follow softmax(d / T)
    wl = workload("tiny_chain").scaled(V=6, B=4000, gamma=1)
    d = logits_inputs(wl, 3)
    rows = d["draft"][:, 0].astype(np.float64) / wl.T
    # all rows differ; pool by probability integral: P(token) under own row
    pr = np.exp(rows - rows.max(1, keepdims=True))
    pr /= pr.sum(1, keepdims=True)
    tok = d["tokens"][:, 1]
    # expected count per token summed over rows vs observed
    exp = pr.sum(0)
    obs = np.bincount(tok, minlength=6)
    assert stats.chisquare(obs, exp).pvalue > 1e-3
