"""Pins of the oracle's greedy verify (temperature 0).

Page 1 §4.3 (first point): at temperature 0, or under greedy decoding, the
probabilistic accept test becomes an exact match position by position.  The
oracle reads a row's law at T = 0 as the point mass on its largest logit
(the smallest index among equal largest ones) and runs the same walk.
Pinned here against hand-worked greedy decoding, never against the
oracle's own formulas:

* a chain keeps the longest prefix of drafts equal to the target's argmax
  tokens and then emits the target's argmax at the first mismatch (or, when
  all match, the argmax of the last row): worked out by hand on small rows;
* ties go to the smallest index;
* a tree node accepts the first child, in order, whose token is the argmax;
* the outputs do not depend on the uniforms (seed, offset);
* the sampling rule at a tiny temperature gives the same outputs when the
  largest logit is well separated (softmax(z / T) is then a point mass to
  double precision), a check between two independent code paths;
* temperatures below zero, NaN or infinite still fail the request.
"""
import numpy as np
import pytest

from oracle import INVALID_ARG, greedy_rows, oracle_reject_sample


def _run(target, draft, tokens, parent=None, T=0.0, seed=3, offset=0):
    target = np.asarray(target, dtype=np.float32)[None]
    draft = np.asarray(draft, dtype=np.float32)[None]
    par = None if parent is None else np.asarray(parent, dtype=np.int32)[None]
    return oracle_reject_sample(target, draft, np.asarray(tokens, np.int32)[None], par,
                                np.array([T], np.float32), seed, offset)


# target rows with argmax 2, 4, 0, 1 (by construction)
TGT = [[0.1, 0.5, 3.0, -1.0, 0.0],
       [1.0, 0.0, -2.0, 0.5, 2.5],
       [4.0, 1.0, 3.5, 0.0, 0.0],
       [0.0, 9.0, 1.0, 8.5, 0.0]]
DFT = [[0.0, 0.0, 1.0, 0.0, 0.0],
       [0.0, 0.0, 0.0, 0.0, 1.0],
       [0.0, 0.0, 0.0, 2.0, 0.0],
       [0.0, 1.0, 0.0, 0.0, 0.0]]


def test_chain_prefix_then_argmax():
    # drafts 2, 4 match the argmax of rows 0 and 1; draft 3 does not match
    # row 2's argmax (0): two accepted, then 0
    r = _run(TGT, DFT, [7, 2, 4, 3])
    assert r["status"][0] == 0 and r["accepted_len"][0] == 2
    assert list(r["out_tokens"][0]) == [2, 4, 0, -1]
    assert list(r["path"][0]) == [0, 1, 2, -1]


def test_chain_all_match_then_bonus_argmax():
    r = _run(TGT, DFT, [7, 2, 4, 0])
    assert r["accepted_len"][0] == 3
    assert list(r["out_tokens"][0]) == [2, 4, 0, 1]


def test_chain_first_mismatch():
    r = _run(TGT, DFT, [7, 1, 4, 0])
    assert r["accepted_len"][0] == 0
    assert list(r["out_tokens"][0]) == [2, -1, -1, -1]


def test_ties_go_to_the_smallest_index():
    z = [[1.0, 5.0, 5.0, 0.0], [0.0, 0.0, 0.0, 0.0]]
    d = [[0.0, 0.0, 1.0, 0.0], [0.0, 0.0, 0.0, 0.0]]
    assert list(greedy_rows(np.array(z))[0]) == [0.0, 1.0, 0.0, 0.0]
    r = _run(z, d, [0, 2])            # 2 ties with 1 but 1 comes first
    assert r["accepted_len"][0] == 0 and r["out_tokens"][0, 0] == 1
    r = _run(z, d, [0, 1])
    assert r["accepted_len"][0] == 1
    assert list(r["out_tokens"][0]) == [1, 0]   # row 1: all equal, index 0


def test_tree_first_matching_child_in_order():
    # root argmax 2; children 1, 2, 3 drafted 3, 2, 2: child 1 is rejected,
    # child 2 accepted (child 3 never tested); node 2 is a leaf: its argmax 4
    z = [[0.0, 1.0, 6.0, 2.0, 0.0],
         [0.0] * 5,
         [0.0, 0.0, 0.0, 1.0, 3.0],
         [0.0] * 5]
    d = [[0.0, 0.0, 0.0, 5.0, 0.0]] + [[0.0] * 5] * 3
    r = _run(z, d, [0, 3, 2, 2], parent=[-1, 0, 0, 0])
    assert r["accepted_len"][0] == 1
    assert list(r["path"][0]) == [0, 2, -1, -1]
    assert list(r["out_tokens"][0]) == [2, 4, -1, -1]
    pr = r["probe"][0]
    assert list(pr[1, :2]) == [0.0, 1.0]      # P(3) = 0, Q(3) = 1 (draft argmax 3)
    assert list(pr[2, :2]) == [1.0, 0.0]      # after the rejection P is still the point mass on 2
    assert list(pr[3]) == [-1.0] * 4
    assert list(pr[2, 2:]) == [1.0, 1.0]


def test_outputs_do_not_depend_on_the_uniforms():
    rng = np.random.default_rng(5)
    z = rng.normal(0, 3, (6, 50)).astype(np.float32)
    d = (z + rng.normal(0, 1, (6, 50))).astype(np.float32)
    toks = np.argmax(z, axis=1)
    toks = np.concatenate([[0], toks[:5]])
    toks[3] = (toks[3] + 1) % 50       # a mismatch at position 3
    ref = _run(z, d, toks, seed=1, offset=0)
    assert ref["accepted_len"][0] == 2
    for seed, off in [(2, 0), (9, 5), (12345, 77)]:
        r = _run(z, d, toks, seed=seed, offset=off)
        for k in ("out_tokens", "path", "accepted_len"):
            assert np.array_equal(r[k], ref[k])
    assert np.isinf(ref["margin"][0])    # no decision is near a threshold


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_temperature_gives_the_same_outputs(seed):
    # rows whose largest logit leads the next by at least 0.5: at T = 1e-3
    # the softmax puts all but e^-500 of its mass on it
    rng = np.random.default_rng(seed)
    M, V = 5, 40
    z = rng.normal(0, 2, (M, V))
    for n in range(M):
        k = rng.integers(V)
        z[n, k] = z[n].max() + 0.5 + rng.random()
    d = z + rng.normal(0, 0.3, (M, V))
    for n in range(M):
        d[n, np.argmax(d[n])] += 0.5
    toks = np.concatenate([[0], np.argmax(z, axis=1)[:M - 1]])
    toks[1 + seed] = np.argmin(z[seed])  # a mismatch, at a different place per seed
    g = _run(z.astype(np.float32), d.astype(np.float32), toks, T=0.0)
    s = _run(z.astype(np.float32), d.astype(np.float32), toks, T=1e-3)
    for k in ("out_tokens", "path", "accepted_len"):
        assert np.array_equal(g[k], s[k]), k


@pytest.mark.parametrize("T", [-1.0, np.nan, np.inf, 1e-40])
def test_bad_temperatures_still_fail(T):
    r = _run(TGT, DFT, [7, 2, 4, 3], T=T)
    assert r["status"][0] == INVALID_ARG and r["accepted_len"][0] == -1
