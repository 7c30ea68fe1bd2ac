"""Pins of the oracle's KV commit (page 2 §3.3 rollback; §5.4 tree path).

* A chain commit moves nothing: only the length changes, to ctx + a + 1.
* A tree commit equals a gather along the accepted path taken from an
  untouched copy of the cache (brute force), for random root-to-node paths.
* A failed request (a = -1) keeps its length and its bytes.
"""
import numpy as np

from oracle import oracle_kv_commit
from synth import random_tree


def _cache(rng, nb=12, Hkv=2, block=16, D=4):
    return rng.normal(size=(nb, Hkv, block, D)), rng.normal(size=(nb, Hkv, block, D))


def test_chain_commit_is_length_update():
    rng = np.random.default_rng(0)
    kc, vc = _cache(rng)
    table = rng.permutation(12).reshape(3, 4).astype(np.int32)
    ctx = np.array([5, 17, 40], dtype=np.int32)
    acc = np.array([0, 3, 4], dtype=np.int32)
    path = np.tile(np.arange(6), (3, 1)).astype(np.int32)
    k2, v2, n2 = oracle_kv_commit(kc, vc, table, ctx, path, acc)
    assert np.array_equal(k2, kc) and np.array_equal(v2, vc)
    assert n2.tolist() == [6, 21, 45]


def test_tree_commit_equals_gather_from_copy():
    rng = np.random.default_rng(1)
    for trial in range(40):
        M = 21
        parent = random_tree(rng, 4, 3, M)
        kc, vc = _cache(rng, nb=8)
        table = rng.permutation(8).reshape(2, 4).astype(np.int32)
        ctx = np.array([rng.integers(0, 30), rng.integers(0, 30)], np.int32)
        path = np.full((2, M), -1, dtype=np.int32)
        acc = np.zeros(2, dtype=np.int32)
        for b in range(2):
            # random root-to-node path
            node, pth = 0, [0]
            while True:
                kids = [c for c in range(M) if parent[c] == node]
                if not kids or rng.random() < 0.25:
                    break
                node = int(rng.choice(kids))
                pth.append(node)
            path[b, :len(pth)] = pth
            acc[b] = len(pth) - 1
        k2, v2, n2 = oracle_kv_commit(kc, vc, table, ctx, path, acc)
        kx, vx = kc.copy(), vc.copy()
        for b in range(2):
            for j in range(1, acc[b] + 1):
                s = ctx[b] + path[b, j]
                d = ctx[b] + j
                kx[table[b, d // 16], :, d % 16] = kc[table[b, s // 16], :, s % 16]
                vx[table[b, d // 16], :, d % 16] = vc[table[b, s // 16], :, s % 16]
        assert np.array_equal(k2, kx) and np.array_equal(v2, vx)
        assert np.array_equal(n2, ctx + acc + 1)


def test_failed_request_untouched():
    rng = np.random.default_rng(2)
    kc, vc = _cache(rng, nb=4)
    table = np.arange(4, dtype=np.int32).reshape(1, 4)
    path = np.array([[0, 3, 5, -1, -1, -1]], dtype=np.int32)
    k2, v2, n2 = oracle_kv_commit(kc, vc, table, np.array([9], np.int32),
                                  path, np.array([-1], np.int32))
    assert np.array_equal(k2, kc) and n2.tolist() == [9]
