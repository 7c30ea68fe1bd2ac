"""Pins of the oracle's filtered verify (top-k / top-p restricted laws).

Page 2 §5.1 asks that target and draft sample by the same rule (its example:
a nucleus-sampling target and a greedy draft drift apart).  The oracle
restricts both laws of every row to the same kind of prefix of the tokens
ordered by logit, largest first (ties: smaller index first): the first k, then
the shortest prefix holding top_p of their mass, renormalised.  Pinned here:

* hand-computed cases of each filter and of the two together, ties included;
* an independent characterisation by brute force over subsets (the kept set
  is the largest-mass set of its size, the lexicographically smallest among
  equal masses; top-p keeps the smallest such set reaching the target);
* reductions: no filter, k >= V and top_p = 1 change nothing; k = 1 is
  greedy decoding (the T = 0 walk), whatever the temperature;
* exact enumeration: drafts drawn from the restricted draft law, every
  accept/reject branch and sample enumerated -- the emitted tokens follow the
  restricted target law exactly (a mistake in how zero-mass tokens are
  tested or drawn breaks it);
* invalid filters fail the request.
"""
import itertools

import numpy as np
import pytest

from oracle import (FILTER_NEAR, INVALID_ARG, filter_law, filter_order, oracle_reject_sample,
                    row_law)
from oracle.reject_sample import children_lists, verify_request
from test_oracle_reject import _node_prefixes, enumerate_outcomes


def _law(vals):
    v = np.asarray(vals, dtype=np.float64)
    return v / v.sum(), np.log(v)


def test_top_k_hand_cases():
    law, z = _law([0.1, 0.5, 0.4])
    out, m = filter_law(law, z, top_k=2)
    assert np.allclose(out, [0.0, 5 / 9, 4 / 9], atol=1e-15) and m == np.inf
    # equal logits: the smaller indices are kept
    z = np.array([1.0, 1.0, 1.0, 0.0])
    law = np.exp(z) / np.exp(z).sum()
    out, _ = filter_law(law, z, top_k=2)
    assert np.allclose(out, [0.5, 0.5, 0.0, 0.0], atol=1e-15)
    assert list(filter_order(np.array([0.0, 2.0, 2.0, 1.0]))) == [1, 2, 3, 0]


def test_top_p_hand_cases():
    law = np.array([0.5, 0.3, 0.2])
    z = np.log(law)
    out, m = filter_law(law, z, top_p=0.7)     # 0.5 < 0.7 <= 0.8
    assert np.allclose(out, [0.625, 0.375, 0.0], atol=1e-15)
    assert abs(m - 0.1 / 0.7) < 1e-12           # 0.8 - 0.7 = 0.1 above, 0.2 below
    out, _ = filter_law(law, z, top_p=0.5)     # the first token alone reaches 0.5
    assert np.allclose(out, [1.0, 0.0, 0.0])
    # an unsorted row: the order is by logit, not by index
    law2 = np.array([0.2, 0.5, 0.3])
    out, _ = filter_law(law2, np.log(law2), top_p=0.75)
    assert np.allclose(out, [0.0, 0.625, 0.375], atol=1e-15)


def test_top_k_then_top_p():
    law = np.array([0.5, 0.3, 0.2])
    z = np.log(law)
    # first two: mass 0.8; 0.9 of it is 0.72, reached by the second token
    out, _ = filter_law(law, z, top_k=2, top_p=0.9)
    assert np.allclose(out, [0.625, 0.375, 0.0], atol=1e-15)
    # 0.6 of 0.8 is 0.48, reached by the first token
    out, _ = filter_law(law, z, top_k=2, top_p=0.6)
    assert np.allclose(out, [1.0, 0.0, 0.0])


def _brute_keep(law, z, k, tp):
    """Kept set by enumeration of subsets (independent of the sort)."""
    V = len(law)

    def best(n, among):
        # the largest-mass n-subset of `among`, lexicographically smallest on ties
        cands = list(itertools.combinations(sorted(among), n))
        key = lambda S: (-round(sum(law[i] for i in S), 12), S)   # noqa: E731
        return min(cands, key=key)

    allv = list(range(V))
    n = V if k <= 0 else min(k, V)
    # equal logits have equal mass, and a larger logit has more mass: the
    # largest-mass n-subset is the top-n prefix (smaller indices on ties)
    K = best(n, allv)
    if tp >= 1.0:
        return set(K)
    target = tp * sum(law[i] for i in K)
    for m in range(1, n + 1):
        S = best(m, K)
        if sum(law[i] for i in S) >= target:
            return set(S)
    return set(K)


def test_filters_match_subset_enumeration():
    rng = np.random.default_rng(5)
    checked = 0
    for trial in range(300):
        V = int(rng.integers(2, 7))
        # integer-valued logits so that ties are frequent
        z = rng.integers(-2, 3, size=V).astype(np.float64)
        law = np.exp(z) / np.exp(z).sum()
        k = int(rng.integers(0, V + 2))
        tp = float(rng.choice([1.0, 0.3, 0.5, 0.65, 0.8, 0.95]))
        out, m = filter_law(law, z, k, tp)
        if m < 1e-9:
            continue                   # a cut exactly at the target: either side is fine
        assert set(np.nonzero(out)[0]) == _brute_keep(law, z, k, tp), (z, k, tp)
        assert abs(out.sum() - 1.0) < 1e-12
        checked += 1
    assert checked > 200


def _batch(rng, B, M, V, tree):
    tgt = rng.normal(0, 2, (B, M, V)).astype(np.float32)
    dft = (tgt + rng.normal(0, 1, (B, M, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, M)).astype(np.int32)
    par = None
    if tree:
        par = np.array([[-1, 0, 0, 1, 1, 2][:M]] * B, np.int32)
    return tgt, dft, tok, par


@pytest.mark.parametrize("tree", [False, True])
def test_no_filter_and_wide_filters_change_nothing(tree):
    rng = np.random.default_rng(8)
    B, M, V = 12, 6, 40
    tgt, dft, tok, par = _batch(rng, B, M, V, tree)
    T = np.full(B, 0.9, np.float32)
    base = oracle_reject_sample(tgt, dft, tok, par, T, 3, 1)
    for k, tp in [(np.zeros(B, np.int32), np.ones(B, np.float32)),
                  (np.full(B, V, np.int32), np.ones(B, np.float32)),
                  (np.full(B, V + 7, np.int32), None)]:
        f = oracle_reject_sample(tgt, dft, tok, par, T, 3, 1, top_k=k, top_p=tp)
        for key in ("out_tokens", "path", "accepted_len"):
            assert np.array_equal(f[key], base[key])
        assert np.allclose(f["probe"], base["probe"])


@pytest.mark.parametrize("tree", [False, True])
def test_top_k_one_is_greedy(tree):
    rng = np.random.default_rng(9)
    B, M, V = 16, 6, 30
    tgt, dft, tok, par = _batch(rng, B, M, V, tree)
    # some drafts are their parent's argmax so that acceptances happen
    for b in range(B):
        for c in range(1, M):
            pn = c - 1 if par is None else par[b, c]
            if (b + c) % 2:
                tok[b, c] = int(np.argmax(tgt[b, pn]))
    g = oracle_reject_sample(tgt, dft, tok, par, np.zeros(B, np.float32), 4, 0)
    f = oracle_reject_sample(tgt, dft, tok, par, np.full(B, 0.7, np.float32), 4, 0,
                             top_k=np.ones(B, np.int32))
    assert (g["accepted_len"] > 0).any()
    for key in ("out_tokens", "path", "accepted_len"):
        assert np.array_equal(f[key], g[key])


def _filtered_tables(rng, V, depth, k, tp):
    p_tab, q_tab = {}, {}
    for L in range(depth + 1):
        for pre in itertools.product(range(V), repeat=L):
            zt = rng.integers(-2, 3, size=V).astype(np.float64)   # ties included
            zd = zt + rng.integers(-1, 2, size=V)
            p_tab[pre] = filter_law(row_law(zt, 1.0), zt, k, tp)[0]
            q_tab[pre] = filter_law(row_law(zd, 1.0), zd, k, tp)[0]
    return p_tab, q_tab


@pytest.mark.parametrize("parent,k,tp", [
    ([-1, 0, 1], 2, 1.0),
    ([-1, 0, 1], 0, 0.7),
    ([-1, 0, 0], 3, 0.8),
    ([-1, 0, 0, 1], 2, 0.9),
])
def test_exact_law_of_filtered_verify(parent, k, tp):
    """Drafts from the restricted draft law; the emitted tokens follow the
    restricted target law exactly."""
    parent = np.asarray(parent)
    M, V = len(parent), 4
    depth = max(len(_node_prefixes(parent, [0] * M)[n]) for n in range(M))
    rng = np.random.default_rng(M * 7 + k)
    p_tab, q_tab = _filtered_tables(rng, V, depth, k, tp)
    kids = children_lists(parent, M)
    law = {}
    for assign in itertools.product(range(V), repeat=M - 1):
        tokens = [0] + list(assign)
        pre = _node_prefixes(parent, tokens)
        w_draft = 1.0
        for c in range(1, M):
            w_draft *= q_tab[pre[parent[c]]][tokens[c]]
        if w_draft == 0.0:
            continue

        def run(ch, pre=pre, tokens=tokens):
            return verify_request(lambda n: p_tab[pre[n]], lambda n: q_tab[pre[n]],
                                  tokens, kids, ch)

        for res, w in enumerate_outcomes(run):
            seq = tuple(res["emitted"])
            ext = [(seq, w_draft * w)]
            while len(ext[0][0]) < depth + 1:
                ext = [(s + (t,), ww * p_tab[s][t]) for s, ww in ext for t in range(V)]
            for s, ww in ext:
                law[s] = law.get(s, 0.0) + ww
    worst = 0.0
    for s in itertools.product(range(V), repeat=depth + 1):
        pr = 1.0
        for i in range(depth + 1):
            pr *= p_tab[s[:i]][s[i]]
        worst = max(worst, abs(law.get(s, 0.0) - pr))
    assert abs(sum(law.values()) - 1.0) < 1e-12
    assert worst < 1e-12
    # the restriction removed something: tokens outside the kept sets never appear
    assert any((p == 0).any() for p in p_tab.values())


def test_filter_margin_is_reported():
    rng = np.random.default_rng(10)
    B, M, V = 6, 4, 50
    tgt, dft, tok, par = _batch(rng, B, M, V, False)
    f = oracle_reject_sample(tgt, dft, tok, par, np.ones(B, np.float32), 2, 0,
                             top_p=np.full(B, 0.9, np.float32))
    assert np.all(np.isfinite(f["flt_margin"])) and np.all(f["flt_margin"] > 0)
    g = oracle_reject_sample(tgt, dft, tok, par, np.ones(B, np.float32), 2, 0)
    assert np.all(np.isinf(g["flt_margin"]))
    assert FILTER_NEAR < 1e-3


def test_invalid_filters_fail_the_request():
    rng = np.random.default_rng(11)
    B, M, V = 5, 3, 20
    tgt, dft, tok, par = _batch(rng, B, M, V, False)
    k = np.array([0, -1, 0, 0, 0], np.int32)
    tp = np.array([1.0, 1.0, 0.0, 1.5, np.nan], np.float32)
    f = oracle_reject_sample(tgt, dft, tok, par, np.ones(B, np.float32), 1, 0,
                             top_k=k, top_p=tp)
    assert list(f["status"]) == [0, INVALID_ARG, INVALID_ARG, INVALID_ARG, INVALID_ARG]
    assert list(f["accepted_len"][1:]) == [-1] * 4
