"""Pins of the oracle's paged-KV append and verify attention.

* Batched masked attention equals token-by-token decoding, where each
  position sees the cached prefix and the K/V decoded before it (page 1 §2.1:
  the causal mask makes the parallel pass exactly match token-by-token
  decoding); for trees, each node equals decoding along its ancestor chain
  (page 3, tree-attention section).  The token-by-token path builds its key
  list explicitly and never forms a mask.
* Closed forms: q = 0 gives the plain mean of the visible values; identical
  keys give the mean as well; a dominant key returns its value; a request
  with no cache sees only the new keys of its ancestors.
* Block tables: the result does not depend on where the blocks live.
* The append: an identity block table makes the paged cache a plain
  reshape; positions ctx .. ctx+M-1 hold the new rows and the rest of the
  last touched block is zero.
* A degenerate tree (every node has one child) is the causal chain.
"""
import numpy as np
import pytest

from oracle import (ancestors_or_self, gather_positions, oracle_kv_append,
                    oracle_verify_attn, oracle_verify_attn_tokenwise)
from synth import kv_inputs_host, random_tree, workload


def _small(seed, B=3, M=5, Hq=4, Hkv=2, D=16, ctx=(0, 7, 33), block=16,
           tree=False):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx[:B], dtype=np.int32)
    need = (ctx + M + block - 1) // block
    nb = int(need.sum()) + 2
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((B, int(need.max()) + 1), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, :need[b]] = perm[off:off + need[b]]
        off += need[b]
    kc = rng.normal(size=(nb, Hkv, block, D))
    vc = rng.normal(size=(nb, Hkv, block, D))
    q = rng.normal(size=(B, M, Hq, D))
    kn = rng.normal(size=(B, M, Hkv, D))
    vn = rng.normal(size=(B, M, Hkv, D))
    parent = None
    if tree:
        parent = np.stack([random_tree(rng, 3, 3, M) for _ in range(B)])
    return dict(q=q, k_cache=kc, v_cache=vc, block_table=table, ctx_lens=ctx,
                k_new=kn, v_new=vn, parent=parent)


@pytest.mark.parametrize("tree", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 1)])
def test_batched_equals_tokenwise(tree, Hq, Hkv):
    a = _small(1, Hq=Hq, Hkv=Hkv, M=9 if tree else 5, tree=tree)
    o1, l1, _, _ = oracle_verify_attn(**a)
    o2, l2 = oracle_verify_attn_tokenwise(**a)
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs(l1 - l2)) < 1e-12


def test_batched_equals_tokenwise_tiny_workload():
    wl = workload("tiny_chain")
    a = kv_inputs_host(wl, seed=0)
    args = dict(q=a["q"], k_cache=a["k_cache"], v_cache=a["v_cache"],
                block_table=a["block_table"], ctx_lens=a["ctx_lens"],
                k_new=a["k_new"], v_new=a["v_new"])
    o1, l1, _, _ = oracle_verify_attn(**args)
    o2, l2 = oracle_verify_attn_tokenwise(**args)
    assert np.max(np.abs(o1 - o2)) < 1e-12


def test_zero_query_gives_mean_of_visible_values():
    a = _small(2, tree=True, M=7)
    a["q"][:] = 0.0
    o, lse, kc, vc = oracle_verify_attn(**a)
    B, M = a["q"].shape[:2]
    Hq, Hkv = a["q"].shape[2], a["k_new"].shape[2]
    for b in range(B):
        ctx = a["ctx_lens"][b]
        Vp = gather_positions(a["v_cache"], a["block_table"][b],
                              np.arange(ctx), 16)
        for i in range(M):
            chain = ancestors_or_self(a["parent"][b], i)
            vis = np.concatenate([Vp, a["v_new"][b, chain]])
            for h in range(Hq):
                g = h // (Hq // Hkv)
                assert np.allclose(o[b, i, h], vis[:, g].mean(0), atol=1e-13)
                assert abs(lse[b, i, h] - np.log(len(vis))) < 1e-13


def test_identical_keys_and_dominant_key():
    a = _small(3, B=1, ctx=(20,), M=4)
    a["k_cache"][:] = 0.5
    a["k_new"][:] = 0.5
    o, _, _, _ = oracle_verify_attn(**a)
    V = gather_positions(a["v_cache"], a["block_table"][0], np.arange(20), 16)
    for i in range(4):
        vis = np.concatenate([V, a["v_new"][0, :i + 1]])
        for h in range(4):
            assert np.allclose(o[0, i, h], vis[:, h // 2].mean(0), atol=1e-13)
    # dominant key: new key of row 0 aligned with the query, scaled large
    b = _small(4, B=1, ctx=(20,), M=1, Hq=2, Hkv=2)
    b["k_new"][0, 0] = 60.0 * b["q"][0, 0]
    o, _, _, _ = oracle_verify_attn(**b)
    assert np.allclose(o[0, 0], b["v_new"][0, 0], atol=1e-9)


def test_empty_cache_single_key():
    a = _small(5, B=1, ctx=(0,), M=1)
    o, lse, _, _ = oracle_verify_attn(**a)
    for h in range(4):
        assert np.allclose(o[0, 0, h], a["v_new"][0, 0, h // 2], atol=1e-14)


def test_block_placement_does_not_matter():
    a = _small(6, tree=True, M=6)
    o1, l1, _, _ = oracle_verify_attn(**a)
    # move every block to a new physical index
    nb = a["k_cache"].shape[0]
    perm = np.random.default_rng(0).permutation(nb)
    kc = np.empty_like(a["k_cache"])
    vc = np.empty_like(a["v_cache"])
    kc[perm] = a["k_cache"]
    vc[perm] = a["v_cache"]
    t = np.where(a["block_table"] >= 0, perm[a["block_table"]], -1)
    b = dict(a, k_cache=kc, v_cache=vc, block_table=t)
    o2, l2, _, _ = oracle_verify_attn(**b)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_degenerate_tree_is_chain():
    a = _small(7, M=5)
    b = dict(a, parent=np.tile(np.arange(-1, 4), (3, 1)))
    o1, _, _, _ = oracle_verify_attn(**a)
    o2, _, _, _ = oracle_verify_attn(**b)
    assert np.array_equal(o1, o2)


def test_append_identity_table_and_tail():
    B, M, Hkv, D, block = 2, 5, 2, 8, 16
    ctx = np.array([3, 27], dtype=np.int32)
    need = (ctx + M + block - 1) // block          # [1, 2]
    table = np.array([[0, -1], [1, 2]], dtype=np.int32)
    rng = np.random.default_rng(8)
    kc = rng.normal(size=(3, Hkv, block, D))
    vc = rng.normal(size=(3, Hkv, block, D))
    kn = rng.normal(size=(B, M, Hkv, D))
    vn = rng.normal(size=(B, M, Hkv, D))
    k2, v2 = oracle_kv_append(kc, vc, table, ctx, kn, vn, block)
    # request 1 owns blocks 1, 2 contiguously: positions t -> block 1 + t//16
    flat = k2[1:3].transpose(0, 2, 1, 3).reshape(2 * block, Hkv, D)
    assert np.array_equal(flat[27:32], kn[1])
    assert np.all(flat[32:] == 0)
    assert np.array_equal(flat[:27], kc[1:3].transpose(0, 2, 1, 3)
                          .reshape(2 * block, Hkv, D)[:27])
    flat0 = v2[0].transpose(1, 0, 2)
    assert np.array_equal(flat0[3:8], vn[0])
    assert np.all(flat0[8:] == 0)
    assert np.array_equal(flat0[:3], vc[0].transpose(1, 0, 2)[:3])
    assert need.tolist() == [1, 2]
