"""Pins of the oracle's probe columns (what each accept test and the draw used).

For every tested node the oracle records P(x) and Q(x) as used in its accept
test (columns 0 and 1); at the node where the draw happened it records the
mass Z of the residual drawn from (1 for a draw from p) and the probability
of the drawn token under the normalised law (columns 2 and 3).  The GPU is
held to these columns, so each one is pinned here against hand-computed
values, never against the oracle's own formulas:

* target and draft rows are built as z = T * ln(w) for hand-chosen
  probability vectors w, so softmax(z / T) = w exactly (up to fp64
  rounding) at any temperature; every expected P, Q, residual mass and
  residual probability below is a rational number worked out by hand from
  the accept rule of page 1 §2.3 / §4.1 (accept x with probability
  min(1, p(x)/q(x))), the residual normalize(max(0, p - q)) of page 3's
  formal definition, and the sibling rule for trees (each rejected child
  turns the working target into the normalised residual of the previous
  one);
* drafted tokens are chosen with p(x) = 0 (rejected whatever the uniform)
  or p(x) >= q(x) (accepted whatever the uniform), so the walk does not
  depend on the uniforms; only the final draw does, and its uniform comes
  from the Philox generator pinned separately by its published
  known-answer vectors.

A plausible recording mistake fails one of these: P recorded before a
sibling's residual update (0.6 instead of 5/6), the first residual's mass
reported instead of the last (0.6 instead of 11/15), or the drawn token's
probability normalised by the wrong mass (0.5 instead of 5/6).
"""
import numpy as np
import pytest

from oracle import oracle_reject_sample, uniforms_for

SEED, OFFSET = 4321, 7


def _logits(w, T):
    w = np.asarray(w, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return T * np.log(w)


def _run(p_rows, q_rows, tokens, parent, T):
    M = len(tokens)
    target = np.stack([_logits(w, T) for w in p_rows])[None]
    draft = np.stack([_logits(w, T) for w in q_rows])[None]
    par = None if parent is None else np.asarray(parent, dtype=np.int32)[None]
    res = oracle_reject_sample(target, draft, np.asarray(tokens, np.int32)[None],
                               par, np.array([T], np.float32), SEED, OFFSET)
    assert res["status"][0] == 0
    assert res["path"].shape == (1, M)
    return res


def _u_smp(node, M):
    return uniforms_for(SEED, OFFSET, 0, M)[1][node]


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_chain_probe_accept_then_certain_reject(T):
    # node 0: p0 = (0.6, 0.4, 0), q0 = (0.1, 0.3, 0.6); draft x1 = 0 has
    #   p >= q, so it is accepted: probe (0.6, 0.1)
    # node 1: p1 = (0, 0.5, 0.5), q1 = (0.5, 0.25, 0.25); draft x2 = 0 has
    #   p = 0, so it is rejected: probe (0, 0.5)
    # the draw at node 1 is from max(0, p1 - q1) = (0, 0.25, 0.25):
    #   Z = 0.5, normalised (0, 0.5, 0.5), so the drawn token has 0.5
    p = [[0.6, 0.4, 0.0], [0.0, 0.5, 0.5], [0.2, 0.3, 0.5]]
    q = [[0.1, 0.3, 0.6], [0.5, 0.25, 0.25], [1 / 3, 1 / 3, 1 / 3]]
    res = _run(p, q, [0, 0, 0], None, T)
    pr = res["probe"][0]
    assert res["accepted_len"][0] == 1
    np.testing.assert_allclose(pr[1, :2], [0.6, 0.1], atol=1e-12)
    np.testing.assert_allclose(pr[2, :2], [0.0, 0.5], atol=1e-12)
    np.testing.assert_allclose(pr[1, 2:], [0.5, 0.5], atol=1e-12)
    assert np.all(pr[0] == -1.0) and np.all(pr[2, 2:] == -1.0)
    u = _u_smp(1, 3)
    assert res["out_tokens"][0, 1] == (1 if u < 0.5 else 2)
    assert res["out_tokens"][0, 0] == 0


def test_chain_probe_all_accepted_bonus():
    # every draft has p(x) >= q(x): all accepted; the bonus comes from p of
    # the last node, so Z = 1 and the drawn token has p2[token]
    p = [[0.5, 0.5, 0.0], [0.1, 0.2, 0.7], [0.25, 0.75, 0.0]]
    q = [[0.4, 0.3, 0.3], [0.3, 0.3, 0.4], [0.5, 0.5, 0.0]]
    res = _run(p, q, [0, 0, 2], None, 1.0)
    pr = res["probe"][0]
    assert res["accepted_len"][0] == 2
    np.testing.assert_allclose(pr[1, :2], [0.5, 0.4], atol=1e-12)
    np.testing.assert_allclose(pr[2, :2], [0.7, 0.4], atol=1e-12)
    u = _u_smp(2, 3)
    tok = 0 if u < 0.25 else 1
    assert res["out_tokens"][0, 2] == tok
    np.testing.assert_allclose(pr[2, 2:], [1.0, [0.25, 0.75][tok]], atol=1e-12)


def test_all_reject_residual_mass_and_drawn_probability():
    # p0 = (0.6, 0.4, 0), q0 = (0.1, 0.3, 0.6), x1 = 2 (p = 0): rejected.
    # max(0, p0 - q0) = (0.5, 0.1, 0): Z = 0.6, normalised (5/6, 1/6, 0)
    p = [[0.6, 0.4, 0.0], [0.3, 0.3, 0.4]]
    q = [[0.1, 0.3, 0.6], [0.3, 0.3, 0.4]]
    res = _run(p, q, [0, 2], None, 1.0)
    pr = res["probe"][0]
    assert res["accepted_len"][0] == 0
    np.testing.assert_allclose(pr[1, :2], [0.0, 0.6], atol=1e-12)
    u = _u_smp(0, 2)
    tok = 0 if u < 5 / 6 else 1
    assert res["out_tokens"][0, 0] == tok
    np.testing.assert_allclose(pr[0, 2:], [0.6, [5 / 6, 1 / 6][tok]], atol=1e-12)


def test_tree_second_child_sees_the_updated_target():
    # root p = (0.6, 0.4, 0), q = (0.1, 0.3, 0.6); children 1 (x = 2) and
    # 2 (x = 0).  Child 1 has p = 0: rejected; the working target becomes
    # (5/6, 1/6, 0).  Child 2 is tested against P(0) = 5/6 >= q(0) = 0.1:
    # accepted, and its probe holds 5/6, not the root's p(0) = 0.6.
    # Child 2 is a leaf: bonus from p of node 2 = (0.2, 0.8, 0).
    p = [[0.6, 0.4, 0.0], [0.5, 0.5, 0.0], [0.2, 0.8, 0.0]]
    q = [[0.1, 0.3, 0.6], [0.5, 0.5, 0.0], [0.5, 0.5, 0.0]]
    res = _run(p, q, [0, 2, 0], [-1, 0, 0], 1.0)
    pr = res["probe"][0]
    assert res["accepted_len"][0] == 1 and list(res["path"][0]) == [0, 2, -1]
    np.testing.assert_allclose(pr[1, :2], [0.0, 0.6], atol=1e-12)
    np.testing.assert_allclose(pr[2, :2], [5 / 6, 0.1], atol=1e-12)
    u = _u_smp(2, 3)
    tok = 0 if u < 0.2 else 1
    assert res["out_tokens"][0, 1] == tok
    np.testing.assert_allclose(pr[2, 2:], [1.0, [0.2, 0.8][tok]], atol=1e-12)
    assert np.all(pr[0] == -1.0)


def test_tree_two_rejections_report_the_last_residual():
    # root p = (0.6, 0.4, 0), q = (0.1, 0.3, 0.6); children 1, 2 and 3.
    # child 1, x = 2: P(2) = 0, rejected; P1 = (5/6, 1/6, 0) (mass 0.6)
    # child 2, x = 2: P1(2) = 0, rejected; max(0, P1 - q) = (11/15, 0, 0),
    #   mass Z2 = 11/15, P2 = (1, 0, 0)
    # child 3, x = 1: P2(1) = 0, rejected; max(0, P2 - q) = (0.9, 0, 0),
    #   mass Z3 = 0.9, P3 = (1, 0, 0)
    # the draw at the root uses P3: Z = 0.9 and the drawn token 0 has 1
    p = [[0.6, 0.4, 0.0]] + [[0.5, 0.5, 0.0]] * 3
    q = [[0.1, 0.3, 0.6]] + [[0.5, 0.5, 0.0]] * 3
    res = _run(p, q, [0, 2, 2, 1], [-1, 0, 0, 0], 1.0)
    pr = res["probe"][0]
    assert res["accepted_len"][0] == 0
    np.testing.assert_allclose(pr[1, :2], [0.0, 0.6], atol=1e-12)
    np.testing.assert_allclose(pr[2, :2], [0.0, 0.6], atol=1e-12)
    np.testing.assert_allclose(pr[3, :2], [0.0, 0.3], atol=1e-12)
    assert res["out_tokens"][0, 0] == 0
    np.testing.assert_allclose(pr[0, 2:], [0.9, 1.0], atol=1e-12)


def test_tree_rejection_then_uncertain_child_uses_updated_mass():
    # root p = (0.6, 0.4, 0), q = (0.1, 0.3, 0.6); child 1 (x = 2) rejected,
    # P1 = (5/6, 1/6, 0); child 2 (x = 1): P1(1) = 1/6 < q(1) = 0.3, accepted
    # iff u < (1/6) / 0.3 = 5/9.  If rejected, max(0, P1 - q) = (11/15, 0, 0)
    # and the root draws token 0 with Z = 11/15.
    p = [[0.6, 0.4, 0.0], [0.5, 0.5, 0.0], [0.5, 0.5, 0.0]]
    q = [[0.1, 0.3, 0.6], [0.5, 0.5, 0.0], [0.5, 0.5, 0.0]]
    res = _run(p, q, [0, 2, 1], [-1, 0, 0], 1.0)
    pr = res["probe"][0]
    np.testing.assert_allclose(pr[2, :2], [1 / 6, 0.3], atol=1e-12)
    u_acc = uniforms_for(SEED, OFFSET, 0, 3)[0][2]
    if u_acc < 5 / 9:
        assert res["accepted_len"][0] == 1 and res["path"][0, 1] == 2
    else:
        assert res["accepted_len"][0] == 0 and res["out_tokens"][0, 0] == 0
        np.testing.assert_allclose(pr[0, 2:], [11 / 15, 1.0], atol=1e-12)


def _closed_form_walk(p, q, xs, u_acc):
    """The root's children tested in order, from a closed form of the
    sequential residual updates (derived here, not the oracle's loop): after
    j rejections the working target is max(0, p - c_j q) / D_j with
    c_0 = 0, D_0 = 1, c_{j+1} = c_j + D_j and D_{j+1} = sum max(0, p -
    c_{j+1} q) -- by induction, max(0, max(0, p - c q) / D - q) equals
    max(0, p - (c + D) q) / D, so the normaliser of that residual is
    sum max(0, p - (c + D) q) / D.  Returns the (P(x), Q(x)) of each tested
    child, the accepted child (or None), and the residual mass of the last
    rejection (Z, the probe's column 2 at the root)."""
    c, D = 0.0, 1.0
    tested, Z = [], 1.0
    for k, x in enumerate(xs):
        P = max(0.0, p[x] - c * q[x]) / D
        tested.append((P, q[x]))
        if u_acc[k + 1] * q[x] < P:
            return tested, k + 1, Z
        c = c + D
        D_next = float(np.maximum(p - c * q, 0.0).sum())
        Z = D_next / D
        D = D_next
    return tested, None, Z


@pytest.mark.parametrize("mode", ["favoured", "mixed"])
@pytest.mark.parametrize("seed", range(6))
def test_tree_many_sibling_rejections_closed_form(seed, mode):
    # a root with seven leaf children; random p and q over 9 tokens with
    # every entry positive, so no residual has zero mass.  "favoured": the
    # drafted tokens are the ones the draft favours most over the target
    # (most often rejected: up to seven residual updates in a row);
    # "mixed": those alternate with tokens from the middle of that order,
    # whose residual probabilities stay positive along the walk
    rng = np.random.default_rng((100 if mode == "favoured" else 200) + seed)
    V, W = 9, 7
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.5)
    q = 0.9 * q + 0.1 / V
    order = np.argsort(-q / p)
    picks = range(W) if mode == "favoured" else (0, 4, 1, 5, 2, 6, 3)
    xs = [int(order[i]) for i in picks]
    leaf = np.full(V, 1.0 / V)
    M = 1 + W
    res = _run([p] + [leaf] * W, [q] + [leaf] * W, [0] + xs, [-1] + [0] * W, 1.0)
    pr = res["probe"][0]
    u_acc = uniforms_for(SEED, OFFSET, 0, M)[0]
    tested, accepted, Z = _closed_form_walk(p, q, xs, u_acc)
    for k, (P, Q) in enumerate(tested):
        np.testing.assert_allclose(pr[k + 1, :2], [P, Q], rtol=1e-10, atol=1e-12)
    if accepted is None:
        assert res["accepted_len"][0] == 0
        np.testing.assert_allclose(pr[0, 2], Z, rtol=1e-10)
    else:
        assert res["accepted_len"][0] == 1 and res["path"][0, 1] == accepted
    # children after the accepted one are not tested
    for k in range(len(tested) + 1, M):
        assert np.all(pr[k, :2] == -1.0)
