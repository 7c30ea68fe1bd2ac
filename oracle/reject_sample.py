"""Accept / reject / resample of speculative decoding, fp64 on the CPU.

What the pages fix, and the readings taken where they are silent:

* Temperature softmax of the target logits z and the draft logits d with one
  shared temperature T: p = softmax(z / T), q = softmax(d / T) (page 1 §3.3
  asks for matching draft and target temperatures).
* Accept draft token x with probability min(1, p(x) / q(x)): accept at once if
  p(x) >= q(x), otherwise with probability p(x) / q(x) (page 1 §2.3 and §4.1;
  page 2 §2.1).  With a uniform u in [0, 1) the test is u * q(x) < p(x).
* Stop at the first rejection and drop the later drafts (page 1 §4.3, third
  point).
* After a rejection, draw the replacement from normalize(max(0, p - q)); when
  every draft was accepted draw the extra (bonus) token from p of the last
  accepted position (page 3, formal definition: g drafts + 1 bonus and the
  residual max(0, pi_t - pi_d); the sentence there attaches the residual to
  the all-accepted case, which contradicts the exactness it claims, so the
  residual is used after a rejection and p for the bonus).
* Tree verify (page 1 §5.3; page 2 §5.4; page 3 tree-attention section): the
  pages give no acceptance rule for several children of one node.  Reading
  taken: children were drafted i.i.d. from q of their parent; they are tested
  in ascending node order; after each rejected child the working target
  becomes P <- normalize(max(0, P - q)); the first accepted child becomes the
  new node (with P = p and q of that node); if every child is rejected, or
  the node is a leaf, one token is drawn from the working P.  A chain is the
  tree in which node i has the single child i + 1.
* Sampling is by inverse CDF in vocabulary order: the token is the smallest k
  with C_k > u * Z, where C is the running sum of the weights and Z their
  total.
* A residual of total mass 0 cannot follow a genuine rejection (a rejection
  implies p(x) < q(x)); it only arises for a drafted token of zero draft
  probability.  Reading taken: the working distribution then falls back to
  the target p of the node.
* Rows containing NaN or +inf, or only -inf, have no distribution: the whole
  request is reported as failed (accepted length -1).  -inf entries are
  allowed and have probability 0.
* Temperature 0 is greedy decoding (page 1 §4.3, first point: at temperature
  0, or under greedy decoding, the probabilistic test becomes an exact match
  position by position).  Reading taken: the law of a row at T = 0 is the
  point mass on its largest logit, the smallest index among equal largest
  ones (the limit of softmax(z / T) as T -> 0 when the maximum is unique);
  the same walk then accepts a draft exactly when it is that token, and
  every draw -- after a rejection or at the end -- is that token, whatever
  the uniforms.  Page 2 §5.1 asks for the same sampling rule on both sides,
  so the draft row's law at T = 0 is its own point mass.
* Filtered sampling (page 2 §5.1: a target that samples from its nucleus,
  top-p, and a draft that samples differently make the two laws drift
  apart, so both sides use one rule).  Reading taken: a request may carry a
  top-k count and a top-p mass; each row's law (target and draft alike) is
  restricted to a prefix of its tokens ordered by logit, largest first, the
  smaller index first among equal logits -- the first k of them (top-k), then
  the shortest prefix of those whose mass reaches top_p times their total
  (top-p) -- and renormalised; the verify walk then runs on the restricted
  laws, so its output follows the restricted target law.  k = 0 and
  top_p = 1 leave a row as it is; at T = 0 the filters change nothing (the
  point mass is the first token of the order).
"""
from __future__ import annotations

import numpy as np

from .uniforms import uniforms_for

INVALID_ARG = 1   # request failed: bad temperature or topology
NONFINITE = 5     # request failed: a row it needs has no distribution
BAD_TOKEN = 6     # request failed: a drafted token outside [0, V)
NEAR = 1e-6       # decisions closer than this to their threshold are flagged
FILTER_NEAR = 1e-5  # top-p cuts whose mass is this close (relative) to the target are flagged


def softmax_rows(logits: np.ndarray, T: float) -> np.ndarray:
    """softmax(z / T) of each row, in fp64, from the given (bf16/fp32) values."""
    z = np.asarray(logits, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp((z - m) / float(T))
    return e / e.sum(axis=-1, keepdims=True)


def greedy_rows(logits: np.ndarray) -> np.ndarray:
    """Point mass on the largest logit of each row (smallest index on ties)."""
    z = np.asarray(logits, dtype=np.float64)
    k = np.argmax(z, axis=-1)          # numpy returns the first maximum
    out = np.zeros_like(z)
    np.put_along_axis(out, k[..., None], 1.0, axis=-1)
    return out


def row_law(logits: np.ndarray, T: float) -> np.ndarray:
    """The law of a row at temperature T: softmax(z / T), or the point mass
    on the largest logit at T = 0."""
    return greedy_rows(logits) if T == 0.0 else softmax_rows(logits, T)


def filter_order(logits: np.ndarray) -> np.ndarray:
    """Token indices by logit, largest first; the smaller index first among
    equal logits."""
    z = np.asarray(logits, dtype=np.float64)
    return np.lexsort((np.arange(z.shape[-1]), -z))


def filter_law(law: np.ndarray, logits: np.ndarray, top_k: int = 0, top_p: float = 1.0):
    """A row's law restricted by top-k and then top-p, renormalised.

    Keeps the first n tokens of filter_order(logits): n = top_k (all when
    top_k is 0 or at least V), then the smallest n' <= n whose running mass
    in that order reaches top_p times the mass of the first n (all n when
    top_p is 1).  Returns (restricted law, margin): margin is the relative
    distance of the top-p target from the running masses on either side of
    the cut (inf without a top-p cut).
    """
    law = np.asarray(law, dtype=np.float64)
    V = law.shape[-1]
    order = filter_order(logits)
    n = V if top_k <= 0 else min(int(top_k), V)
    margin = np.inf
    if top_p < 1.0:
        c = np.cumsum(law[order[:n]])
        target = float(top_p) * c[-1]
        cut = int(np.searchsorted(c, target, side="left")) + 1
        cut = min(cut, n)
        above = c[cut - 1] - target
        below = target - (c[cut - 2] if cut >= 2 else 0.0)
        margin = min(abs(above), abs(below)) / target
        n = cut
    out = np.zeros_like(law)
    keep = order[:n]
    out[keep] = law[keep]
    return out / out.sum(), margin


def row_has_distribution(row: np.ndarray) -> bool:
    row = np.asarray(row, dtype=np.float64)
    if np.isnan(row).any() or np.isposinf(row).any():
        return False
    return bool(np.isfinite(row).any())


def inverse_cdf(weights: np.ndarray, u: float, tol: float = NEAR):
    """Smallest k with C_k > u * Z (C = running sum of weights, Z = total).

    Returns (k, distance, band): distance = min |u - t| over the two CDF
    thresholds t = C_{k-1}/Z, C_k/Z that bracket u; band = (k_lo, k_hi), the
    index range of tokens whose CDF interval meets [u - tol, u + tol] (the
    tokens any draw within tol of u could select).
    """
    w = np.asarray(weights, dtype=np.float64)
    C = np.cumsum(w)
    Z = C[-1]
    k = int(np.searchsorted(C, u * Z, side="right"))
    k = min(k, C.shape[0] - 1)
    lo = C[k - 1] / Z if k > 0 else 0.0
    hi = C[k] / Z
    k_lo = int(np.searchsorted(C, (u - tol) * Z, side="right"))
    k_hi = int(np.searchsorted(C, (u + tol) * Z, side="right"))
    k_lo = min(max(k_lo, 0), C.shape[0] - 1)
    k_hi = min(max(k_hi, 0), C.shape[0] - 1)
    return k, min(abs(u - lo), abs(hi - u)), (k_lo, k_hi)


class UniformChooser:
    """Decisions driven by one request's counter-based uniforms."""

    def __init__(self, u_acc: np.ndarray, u_smp: np.ndarray, exact: bool = False):
        self.u_acc = u_acc
        self.u_smp = u_smp
        self.exact = exact           # point-mass laws: no decision is near a threshold
        self.acc_margin = np.inf     # smallest |u - p/q| over the accept tests
        self.smp_margin = np.inf     # |u - nearest CDF step| of the draw
        self.band = None             # tokens a draw within NEAR could select

    @property
    def min_margin(self):
        return min(self.acc_margin, self.smp_margin)

    def accept(self, node: int, P_x: float, Q_x: float) -> bool:
        u = self.u_acc[node]
        if Q_x > 0.0 and not self.exact:
            self.acc_margin = min(self.acc_margin, abs(u - P_x / Q_x))
        return u * Q_x < P_x

    def sample(self, node: int, weights: np.ndarray) -> int:
        k, dist, band = inverse_cdf(weights, self.u_smp[node])
        if not self.exact:
            self.smp_margin = min(self.smp_margin, dist)
        self.band = (k, k) if self.exact else band
        return k


def valid_topology(parent: np.ndarray) -> bool:
    """parent[0] = -1 and 0 <= parent[n] < n for n >= 1."""
    if parent[0] != -1:
        return False
    n = np.arange(1, len(parent))
    return bool(np.all((parent[1:] >= 0) & (parent[1:] < n)))


def children_lists(parent: np.ndarray | None, M: int):
    kids = [[] for _ in range(M)]
    for c in range(1, M):
        par = c - 1 if parent is None else int(parent[c])
        kids[par].append(c)
    return kids


def verify_request(p_row, q_row, tokens, children, chooser):
    """The verify walk of one request.

    p_row(n), q_row(n): normalized fp64 target / draft distributions of node n
    (the distributions over n's children).  tokens[c]: drafted token of node c.
    children[n]: child node indices of n in ascending order.
    chooser: object with accept(node, P_x, Q_x) -> bool and
             sample(node, weights) -> token.

    Returns dict(path, emitted, final, tested, Z, p_sampled):
      path      nodes on the accepted path, starting with the root 0
      emitted   accepted tokens followed by the one sampled token
      final     node at which the sample was drawn
      tested    {child: (P(x_c), Q(x_c))} as used in each accept test
      Z         residual mass normalizing the sampling distribution (1 for a
                bonus draw from p)
      p_sampled probability of the sampled token under that distribution
    """
    node = 0
    path = [0]
    emitted = []
    tested = {}
    while True:
        p_node = p_row(node)
        P = p_node
        Z = 1.0
        accepted = None
        if children[node]:
            Q = q_row(node)
            for c in children[node]:
                x = int(tokens[c])
                tested[c] = (float(P[x]), float(Q[x]))
                if chooser.accept(c, float(P[x]), float(Q[x])):
                    accepted = c
                    break
                r = np.maximum(P - Q, 0.0)
                Z = float(r.sum())
                P = r / Z if Z > 0.0 else p_node
                if Z <= 0.0:
                    Z = 1.0
        if accepted is None:
            tok = chooser.sample(node, P)
            emitted.append(tok)
            return dict(path=path, emitted=emitted, final=node, tested=tested,
                        Z=Z, p_sampled=float(P[tok] / P.sum()))
        path.append(accepted)
        emitted.append(int(tokens[accepted]))
        node = accepted


def oracle_reject_sample(target, draft, tokens, parent, temperature, seed,
                         offset, b_base=0, top_k=None, top_p=None):
    """Verify decisions for a batch.

    target, draft : [B, M, V] logits (row n = distribution over n's children)
    tokens        : [B, M] drafted tokens (tokens[b, 0] ignored)
    parent        : [B, M] parent indices (parent[b, 0] = -1) or None (chain)
    temperature   : [B] fp32 values: positive normal finite, or 0 (greedy)
    seed, offset  : Philox key word and counter word 2; b_base + b is word 1
    top_k, top_p  : [B] int32 / fp32 per-request filters, or None (top_k 0
                    and top_p 1 filter nothing); top_k >= 0 and
                    0 < top_p <= 1, else the request fails (INVALID_ARG)

    Returns dict of numpy arrays:
      out_tokens [B, M] int32 (emitted tokens, then -1)
      path       [B, M] int32 (accepted path node indices, then -1)
      accepted_len [B] int32 (-1 for a failed request)
      probe      [B, M, 4] float64: per tested node (P(x), Q(x)); at the final
                 node (Z, probability of the sampled token); -1 elsewhere
      margin     [B] float64: smallest |u - threshold| over the request's
                 decisions (draws closer than 1e-6 are 'near threshold')
      acc_margin [B] float64: the same over the accept tests only
      smp_margin [B] float64: the same for the final draw only
      band       [B, 2] int32: token index range a draw within 1e-6 of u
                 could have selected (the final draw)
      flt_margin [B] float64: smallest relative margin of a top-p cut over
                 the rows the walk used (inf without one); below FILTER_NEAR
                 the kept set is near its threshold
      status     [B] int32: 0, INVALID_ARG, NONFINITE or BAD_TOKEN
    Failed requests (status != 0) keep accepted_len -1 and -1 rows.
    """
    target = np.asarray(target)
    draft = np.asarray(draft)
    B, M, V = target.shape
    out_tokens = np.full((B, M), -1, dtype=np.int32)
    path_out = np.full((B, M), -1, dtype=np.int32)
    acc = np.full(B, -1, dtype=np.int32)
    probe = np.full((B, M, 4), -1.0, dtype=np.float64)
    margin = np.full(B, np.inf, dtype=np.float64)
    acc_margin = np.full(B, np.inf, dtype=np.float64)
    smp_margin = np.full(B, np.inf, dtype=np.float64)
    band = np.full((B, 2), -1, dtype=np.int32)
    flt_margin = np.full(B, np.inf, dtype=np.float64)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        par = None if parent is None else np.asarray(parent[b])
        kids = children_lists(par, M)
        T = float(np.float32(temperature[b]))
        k = 0 if top_k is None else int(top_k[b])
        tp = 1.0 if top_p is None else float(np.float32(top_p[b]))
        # temperature must be 0 (greedy) or a positive, normal, finite fp32 value
        t_ok = T == 0.0 or (T >= float(np.finfo(np.float32).tiny) and np.isfinite(T))
        f_ok = k >= 0 and tp > 0.0 and tp <= 1.0     # NaN fails both comparisons
        if not t_ok or not f_ok or (par is not None and not valid_topology(par)):
            status[b] = INVALID_ARG
            continue
        if np.any((tokens[b, 1:] < 0) | (tokens[b, 1:] >= V)):
            status[b] = BAD_TOKEN
            continue
        needed = [target[b, n] for n in range(M)]
        needed += [draft[b, n] for n in range(M) if kids[n]]
        if not all(row_has_distribution(r) for r in needed):
            status[b] = NONFINITE
            continue
        u_acc, u_smp = uniforms_for(seed, offset, b_base + b, M)
        chooser = UniformChooser(u_acc, u_smp, exact=(T == 0.0))
        fm = [np.inf]

        def law(rows, n, b=b, T=T, k=k, tp=tp, fm=fm):
            base = row_law(rows[b, n], T)
            if T == 0.0 or (k == 0 and tp >= 1.0):
                return base
            out, m = filter_law(base, rows[b, n], k, tp)
            fm[0] = min(fm[0], m)
            return out

        res = verify_request(lambda n: law(target, n), lambda n: law(draft, n),
                             tokens[b], kids, chooser)
        flt_margin[b] = fm[0]
        a = len(res["path"]) - 1
        acc[b] = a
        path_out[b, :a + 1] = res["path"]
        out_tokens[b, :a + 1] = res["emitted"]
        for c, (px, qx) in res["tested"].items():
            probe[b, c, 0] = px
            probe[b, c, 1] = qx
        probe[b, res["final"], 2] = res["Z"]
        probe[b, res["final"], 3] = res["p_sampled"]
        margin[b] = chooser.min_margin
        acc_margin[b] = chooser.acc_margin
        smp_margin[b] = chooser.smp_margin
        band[b] = chooser.band
    return dict(out_tokens=out_tokens, path=path_out, accepted_len=acc,
                probe=probe, margin=margin, acc_margin=acc_margin,
                smp_margin=smp_margin, band=band, flt_margin=flt_margin,
                status=status)
