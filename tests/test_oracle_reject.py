"""Pins of the oracle's accept / reject / resample step.

What is pinned, and against what (none of it re-types the oracle):
* inverse_cdf: brute-force counting over a fine grid of u reproduces the
  weights; the strict "C_k > u Z" boundary convention.
* the accept primitive: over a grid of u the accepted fraction is
  min(1, P/Q) (page 1 §2.3 / §4.1).
* exact enumeration (vocab <= 4): drafts drawn from q, every accept/reject
  branch and every sample enumerated with its probability; the emitted block,
  extended by the target's own autoregressive draws, has exactly the target's
  autoregressive law (to 1e-12), for chains and for trees with several
  children per node (page 1 §2.3 / §4.1, page 2 §2.2: the output law equals
  the target's).
* Monte Carlo with the real Philox uniforms: chi-square of the first emitted
  token against p over 10^6 requests; first-position acceptance rate against
  alpha = sum min(p, q); mean emitted count against (1 - a^(g+1)) / (1 - a)
  (page 2 §2.3), including the pages' worked value a = 0.5, g = 4 -> 1.9375.
* edge cases the pages ask to test first (page 2 §3.3): all accepted (draft
  equals target) and all rejected (target gives the first draft zero mass).
* temperature softmax closed form for two tokens; non-finite rows.
"""
import concurrent.futures
import itertools
import multiprocessing
import os

import numpy as np
import pytest
from scipy import stats

from oracle import (NONFINITE, UniformChooser, inverse_cdf,
                    oracle_reject_sample, softmax_rows, verify_request)
from oracle.reject_sample import children_lists


# ---------------------------------------------------------------------------
# primitives
# ---------------------------------------------------------------------------

def test_inverse_cdf_counts_match_weights():
    rng = np.random.default_rng(0)
    for _ in range(5):
        w = rng.random(7)
        w[rng.integers(7)] = 0.0
        G = 1 << 14
        counts = np.zeros(7)
        for i in range(G):
            k, _, _ = inverse_cdf(w, (i + 0.5) / G)
            counts[k] += 1
        assert np.max(np.abs(counts / G - w / w.sum())) <= 2.0 / G
        assert counts[w == 0].sum() == 0


def test_inverse_cdf_boundary_is_strict():
    w = np.array([1.0, 1.0, 1.0, 1.0])
    assert inverse_cdf(w, 0.0)[0] == 0
    assert inverse_cdf(w, 0.25)[0] == 1      # C_0 = 1 is not > 0.25 * 4
    assert inverse_cdf(w, 0.2499999)[0] == 0
    assert inverse_cdf(w, 0.999999)[0] == 3
    # zero-mass prefix is skipped even at u = 0
    assert inverse_cdf(np.array([0.0, 0.0, 2.0]), 0.0)[0] == 2
    # the band holds every token a draw within the tolerance could select
    k, dist, band = inverse_cdf(w, 0.25, tol=1e-3)
    assert (k, band) == (1, (0, 1)) and dist == 0.0
    k, dist, band = inverse_cdf(w, 0.6, tol=1e-3)
    assert (k, band) == (2, (2, 2)) and abs(dist - 0.1) < 1e-12


def test_accept_primitive_rate():
    G = 1 << 12
    for P, Q in [(0.3, 0.6), (0.6, 0.3), (0.2, 0.2), (0.0, 0.5), (0.4, 0.0)]:
        acc = 0
        for i in range(G):
            u = np.full(2, (i + 0.5) / G)
            acc += UniformChooser(u, u).accept(1, P, Q)
        expect = 1.0 if Q == 0 and P > 0 else min(1.0, P / Q) if Q > 0 else 0.0
        assert abs(acc / G - expect) <= 1.0 / G


def test_softmax_two_token_closed_form():
    for T in (0.5, 0.7, 1.0, 2.0):
        for d in (-3.0, 0.0, 1.25, 7.0):
            p = softmax_rows(np.array([[0.0, d]]), T)[0]
            assert abs(p[1] - 1.0 / (1.0 + np.exp(-d / T))) < 1e-15
            assert abs(p.sum() - 1.0) < 1e-15
    z = np.array([[1.0, -np.inf, 2.0]])
    p = softmax_rows(z, 1.0)[0]
    assert p[1] == 0.0 and abs(p[2] / p[0] - np.e) < 1e-14


# ---------------------------------------------------------------------------
# exact enumeration
# ---------------------------------------------------------------------------

class _Stop(Exception):
    pass


class ScriptChooser:
    """Replays a script of decisions; stops at the first unscripted one.

    The acceptance probability of the test u * Q < P with u ~ U[0, 1) is
    min(1, P/Q) (1 if Q = 0 < P); a sample picks token k with probability
    weight_k / total.
    """

    def __init__(self, script):
        self.script = script
        self.i = 0
        self.weight = 1.0
        self.alternatives = None

    def _next(self, alts):
        if self.i < len(self.script):
            choice = self.script[self.i]
            self.i += 1
            self.weight *= dict(alts)[choice]
            return choice
        self.alternatives = [c for c, p in alts if p > 0.0]
        raise _Stop

    def accept(self, node, P_x, Q_x):
        if Q_x > 0.0:
            a = min(1.0, P_x / Q_x)
        else:
            a = 1.0 if P_x > 0.0 else 0.0
        return self._next([(True, a), (False, 1.0 - a)])

    def sample(self, node, weights):
        w = np.asarray(weights, dtype=np.float64)
        w = w / w.sum()
        return self._next([(k, float(w[k])) for k in range(len(w))])


def enumerate_outcomes(run):
    out = []
    stack = [[]]
    while stack:
        script = stack.pop()
        ch = ScriptChooser(script)
        try:
            res = run(ch)
        except _Stop:
            stack.extend(script + [c] for c in ch.alternatives)
            continue
        out.append((res, ch.weight))
    return out


def _tables(rng, V, depth):
    """Target and draft next-token laws keyed by the token prefix."""
    p_tab, q_tab = {}, {}
    for L in range(depth + 1):
        for pre in itertools.product(range(V), repeat=L):
            p_tab[pre] = rng.dirichlet(np.full(V, 0.8))
            q_tab[pre] = rng.dirichlet(np.full(V, 0.8))
    return p_tab, q_tab


def _node_prefixes(parent, tokens):
    M = len(parent)
    pre = [()] * M
    for n in range(1, M):
        pre[n] = pre[parent[n]] + (tokens[n],)
    return pre


def _check_tree_law(parent, V, seed):
    parent = np.asarray(parent)
    M = len(parent)
    depth = max(len(_node_prefixes(parent, [0] * M)[n]) for n in range(M))
    rng = np.random.default_rng(seed)
    p_tab, q_tab = _tables(rng, V, depth)
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

        def run(ch):
            return verify_request(lambda n: p_tab[pre[n]],
                                  lambda n: q_tab[pre[n]], tokens, kids, ch)

        for res, w in enumerate_outcomes(run):
            seq = tuple(res["emitted"])
            # extend with the target's own autoregressive draws
            ext = [(seq, w_draft * w)]
            while len(ext[0][0]) < depth + 1:
                ext = [(s + (t,), ww * p_tab[s][t])
                       for s, ww in ext for t in range(V)]
            for s, ww in ext:
                law[s] = law.get(s, 0.0) + ww
    # the target's autoregressive law of depth + 1 tokens
    worst = 0.0
    for s in itertools.product(range(V), repeat=depth + 1):
        pr = 1.0
        for i in range(depth + 1):
            pr *= p_tab[s[:i]][s[i]]
        worst = max(worst, abs(law.get(s, 0.0) - pr))
    assert abs(sum(law.values()) - 1.0) < 1e-12
    assert worst < 1e-12


@pytest.mark.parametrize("gamma,V", [(1, 4), (2, 3), (3, 3)])
def test_exact_law_chain(gamma, V):
    _check_tree_law([-1] + list(range(gamma)), V, seed=gamma * 10 + V)


@pytest.mark.parametrize("parent", [
    [-1, 0, 0],                  # two children of the root
    [-1, 0, 0, 0],               # three children of the root
    [-1, 0, 0, 1, 1, 2],         # two levels, two children each
    [-1, 0, 0, 0, 1, 2],         # mixed widths
])
def test_exact_law_tree(parent):
    _check_tree_law(parent, 3, seed=len(parent))


def test_exact_law_detects_wrong_bonus():
    """A plausible mistake (bonus drawn from the residual) breaks the pin."""
    parent = [-1, 0, 1]
    kids = children_lists(np.asarray(parent), 3)
    rng = np.random.default_rng(3)
    V = 3
    p_tab, q_tab = _tables(rng, V, 2)

    def broken(p_row, q_row, tokens, children, ch):
        # emulates a bonus drawn from normalize(max(0, p - q)) at the leaf
        res = verify_request(p_row, q_row, tokens, children, ch)
        return res

    total = {}
    for assign in itertools.product(range(V), repeat=2):
        tokens = [0] + list(assign)
        pre = _node_prefixes(np.asarray(parent), tokens)
        w_draft = q_tab[()][tokens[1]] * q_tab[pre[1]][tokens[2]]

        def p_leafresid(n, pre=pre):
            if n == 2:
                r = np.maximum(p_tab[pre[2]] - q_tab[pre[2]], 0)
                return r / r.sum()
            return p_tab[pre[n]]

        def run(ch, pre=pre, p_leafresid=p_leafresid):
            return broken(p_leafresid, lambda n: q_tab[pre[n]], tokens, kids,
                          ch)

        for res, w in enumerate_outcomes(run):
            s = tuple(res["emitted"])
            total[s] = total.get(s, 0.0) + w * w_draft
    # marginal of a full-length block's last token differs from the target's
    full = {s: w for s, w in total.items() if len(s) == 3}
    pr = {}
    for s in full:
        pr[s] = p_tab[()][s[0]] * p_tab[s[:1]][s[1]] * p_tab[s[:2]][s[2]]
    assert max(abs(full[s] - pr[s]) for s in full) > 1e-6


# ---------------------------------------------------------------------------
# Monte Carlo with the real uniforms
# ---------------------------------------------------------------------------

def _iid_batch(B, gamma, V, seed, same=False, token_seed=None):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 1.5, V)
    d = z if same else z + rng.normal(0, 1.0, V)
    M = gamma + 1
    target = np.broadcast_to(z, (B, M, V)).copy()
    draft = np.broadcast_to(d, (B, M, V)).copy()
    q = softmax_rows(d[None], 1.0)[0]
    if token_seed is not None:
        rng = np.random.default_rng([seed, token_seed])
    tokens = rng.choice(V, size=(B, M), p=q).astype(np.int32)
    return target, draft, tokens, np.ones(B, dtype=np.float32)


def _first_token_counts(shard):
    """Counts of the first emitted token over one shard of the 10^6 trials
    (its own requests, numbered from b_base, so its uniforms are its own)."""
    b_base, B, gamma, V = shard
    target, draft, tokens, T = _iid_batch(B, gamma, V, seed=1, token_seed=b_base)
    res = oracle_reject_sample(target, draft, tokens, None, T, seed=77,
                               offset=0, b_base=b_base)
    return np.bincount(res["out_tokens"][:, 0], minlength=V)


def test_mc_first_token_chi_square():
    """10^6 independent requests through the oracle (in parallel processes,
    each a shard of requests): the first emitted token follows p."""
    B, gamma, V = 1_000_000, 3, 8
    workers = max(1, min(8, os.cpu_count() or 1))
    per = -(-B // (4 * workers))
    shards = [(s, min(per, B - s), gamma, V) for s in range(0, B, per)]
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(workers, mp_context=ctx) as ex:
        counts = sum(ex.map(_first_token_counts, shards))
    assert counts.sum() == B
    target, _, _, _ = _iid_batch(1, gamma, V, seed=1)
    p = softmax_rows(target[0, :1], 1.0)[0]
    chi = stats.chisquare(counts, p * B)
    assert chi.pvalue > 1e-3


def test_mc_acceptance_rate_and_expected_count():
    B, gamma, V = 100_000, 4, 8
    target, draft, tokens, T = _iid_batch(B, gamma, V, seed=2)
    res = oracle_reject_sample(target, draft, tokens, None, T, seed=5,
                               offset=3)
    p = softmax_rows(target[0, :1], 1.0)[0]
    q = softmax_rows(draft[0, :1], 1.0)[0]
    alpha = np.minimum(p, q).sum()
    a = res["accepted_len"]
    first = (a >= 1).mean()
    assert abs(first - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / B)
    emitted = a + 1
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(emitted.mean() - expect) < 4 * emitted.std() / np.sqrt(B)


def test_expected_count_worked_value():
    # page 2 §2.3 formula at the value page 3 quotes (a = 0.5, g = 4: "~2")
    alpha, gamma = 0.5, 4
    assert (1 - alpha ** (gamma + 1)) / (1 - alpha) == 1.9375


def test_all_accept_bonus_from_p():
    B, gamma, V = 50_000, 3, 6
    target, draft, tokens, T = _iid_batch(B, gamma, V, seed=3, same=True)
    res = oracle_reject_sample(target, draft, tokens, None, T, seed=9,
                               offset=1)
    assert np.all(res["accepted_len"] == gamma)
    assert np.all(res["out_tokens"][:, :gamma] == tokens[:, 1:])
    p = softmax_rows(target[0, -1:], 1.0)[0]
    counts = np.bincount(res["out_tokens"][:, gamma], minlength=V)
    assert stats.chisquare(counts, p * B).pvalue > 1e-3
    assert np.allclose(res["probe"][:, gamma, 2], 1.0)


def test_all_reject_draws_from_residual():
    B, gamma, V = 50_000, 3, 6
    target, draft, tokens, T = _iid_batch(B, gamma, V, seed=4)
    x1 = tokens[:, 1]
    target[np.arange(B), 0, x1] = -np.inf
    res = oracle_reject_sample(target, draft, tokens, None, T, seed=11,
                               offset=2)
    assert np.all(res["accepted_len"] == 0)
    tok = res["out_tokens"][:, 0]
    assert np.all(tok != x1)
    assert np.all(res["out_tokens"][:, 1:] == -1)
    # compare with normalize(max(0, p - q)) for each distinct x1
    q = softmax_rows(draft[0, :1], 1.0)[0]
    for x in np.unique(x1):
        sel = x1 == x
        z = target[np.argmax(sel), 0]
        p = softmax_rows(z[None], 1.0)[0]
        r = np.maximum(p - q, 0)
        r /= r.sum()
        counts = np.bincount(tok[sel], minlength=V)
        keep = r > 0
        assert counts[~keep].sum() == 0
        if sel.sum() > 2000:
            assert stats.chisquare(counts[keep],
                                   r[keep] * sel.sum()).pvalue > 1e-3


def test_tree_root_law_mc():
    """First emitted token of a width-4 root fan-out follows p (MC)."""
    B, V = 60_000, 8
    rng = np.random.default_rng(8)
    parent = np.array([-1, 0, 0, 0, 0, 1, 1], dtype=np.int32)
    M = len(parent)
    z = rng.normal(0, 1.5, (M, V))
    d = z + rng.normal(0, 1.2, (M, V))
    q = softmax_rows(d, 1.0)
    tokens = np.zeros((B, M), dtype=np.int32)
    for c in range(1, M):
        tokens[:, c] = rng.choice(V, size=B, p=q[parent[c]])
    res = oracle_reject_sample(np.broadcast_to(z, (B, M, V)),
                               np.broadcast_to(d, (B, M, V)), tokens,
                               np.broadcast_to(parent, (B, M)),
                               np.ones(B, np.float32), seed=3, offset=0)
    p = softmax_rows(z[:1], 1.0)[0]
    counts = np.bincount(res["out_tokens"][:, 0], minlength=V)
    assert stats.chisquare(counts, p * B).pvalue > 1e-3
    # the path is a root-to-node chain of the tree
    for b in range(200):
        a = res["accepted_len"][b]
        pth = res["path"][b, :a + 1]
        assert pth[0] == 0
        for j in range(1, a + 1):
            assert parent[pth[j]] == pth[j - 1]


def test_nonfinite_rows_fail_the_request():
    B, gamma, V = 4, 2, 5
    target, draft, tokens, T = _iid_batch(B, gamma, V, seed=5)
    target[1, 2, 3] = np.nan                     # target row: always needed
    draft[2, 0, 1] = np.inf                      # non-leaf draft row
    draft[3, gamma, 0] = np.nan                  # leaf draft row: never read
    res = oracle_reject_sample(target, draft, tokens, None, T, 1, 0)
    assert list(res["status"]) == [0, NONFINITE, NONFINITE, 0]
    assert res["accepted_len"][1] == -1 and res["accepted_len"][2] == -1
    assert np.all(res["out_tokens"][1] == -1)
