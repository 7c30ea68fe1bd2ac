"""Workload shapes and seeded input generators.

The pages that describe the method measure on unnamed chat / code /
summarisation traffic with 7B/13B-class targets and 32k-152k vocabularies
(page "推测解码的工程真相 2026", tree-attention section; page 1 §6).  No public
suite is named, so the inputs here are synthetic stand-ins with those shapes:

* target logits  z ~ N(0, sigma^2), draft logits d = z + N(0, noise^2), both
  rounded to bf16 (kept in fp32 for the tiny workload);
* draft tokens drawn from q = softmax(d / T) of their parent row;
* queries, new keys/values and cached keys/values ~ N(0, 1), rounded to bf16
  (fp32 for the tiny workload);
* a paged KV cache [num_blocks, Hkv, block, D] whose block tables are a seeded
  random permutation of the physical blocks;
* for the tree workloads, a random ancestor-closed subtree (64 nodes of the
  full depth-4 width-4 tree; 128 nodes of the depth-4 width-8 tree), numbered
  in BFS order.

Draft tokens are drawn with the Gumbel-max trick (argmax of d/T plus
independent standard Gumbel noise), which samples softmax(d/T) exactly without
evaluating it, so no softmax or inverse-CDF arithmetic lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK = 16


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    sigma: float
    noise: float
    T: float
    Hq: int
    Hkv: int
    D: int
    ctx: tuple                     # ("fixed", n) or ("uniform", lo, hi)
    dtype: str = "bf16"            # element type of logits and of q/k/v/cache
    tree_width: int = 0            # 0 = linear chain
    tree_nodes: int = 0            # nodes including the root (tree only)
    layers: int = 1
    block: int = BLOCK
    extra: dict = field(default_factory=dict)

    @property
    def is_tree(self) -> bool:
        return self.tree_width > 0

    @property
    def M(self) -> int:
        """Query rows per request: pending root + gamma drafts, or tree nodes."""
        return self.tree_nodes if self.is_tree else self.gamma + 1

    def scaled(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The synthetic workloads, named by what they are.
WORKLOADS = {
    "tiny_chain": Workload(
        name="tiny_chain", B=1, gamma=4, V=32, sigma=2.0, noise=0.5, T=1.0,
        Hq=4, Hkv=4, D=64, ctx=("fixed", 128), dtype="f32"),
    "chain_7b": Workload(
        name="chain_7b", B=8, gamma=5, V=32000, sigma=3.0, noise=1.0, T=0.8,
        Hq=32, Hkv=32, D=128, ctx=("fixed", 2048)),
    "chain_gqa_128k": Workload(
        name="chain_gqa_128k", B=32, gamma=8, V=128256, sigma=3.0, noise=0.7,
        T=0.7, Hq=32, Hkv=8, D=128, ctx=("uniform", 1024, 8192)),
    "tree_64": Workload(
        name="tree_64", B=16, gamma=4, V=32000, sigma=3.0, noise=1.0, T=1.0,
        Hq=32, Hkv=32, D=128, ctx=("fixed", 4096), tree_width=4,
        tree_nodes=64),
    # a wide tree past 64 nodes (page "推测解码的工程真相 2026", tree-attention
    # section: widths 6 and 8, batch x width kept at 256): 128 nodes grown in
    # the full depth-4 width-8 tree, 32 requests x width 8 = 256
    "tree_wide_128": Workload(
        name="tree_wide_128", B=32, gamma=4, V=32000, sigma=3.0, noise=1.0, T=1.0,
        Hq=32, Hkv=32, D=128, ctx=("fixed", 4096), tree_width=8,
        tree_nodes=128),
    "stress_gqa_152k": Workload(
        name="stress_gqa_152k", B=128, gamma=4, V=152064, sigma=3.0,
        noise=1.5, T=1.0, Hq=64, Hkv=8, D=128, ctx=("uniform", 4096, 32768)),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


# ---------------------------------------------------------------------------
# bf16 helpers (round-to-nearest-even on the upper 16 bits of an fp32)
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    # keep infinities / NaNs as they are
    special = (u & 0x7F800000) == 0x7F800000
    r = np.where(special, u >> 16, r)
    return r.astype(np.uint16)


def bf16_from_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Values of x rounded to bf16, returned as fp32."""
    return bf16_from_bits(bf16_bits(x))


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32)
    return bf16_round(x) if dtype == "bf16" else x


# ---------------------------------------------------------------------------
# structure
# ---------------------------------------------------------------------------

def context_lengths(wl: Workload, seed: int) -> np.ndarray:
    rng = np.random.default_rng([seed, 11])
    if wl.ctx[0] == "fixed":
        return np.full(wl.B, wl.ctx[1], dtype=np.int32)
    lo, hi = wl.ctx[1], wl.ctx[2]
    return rng.integers(lo, hi + 1, size=wl.B).astype(np.int32)


def random_tree(rng: np.random.Generator, depth: int, width: int,
                n_nodes: int) -> np.ndarray:
    """Parent array (BFS numbering, parent[0] = -1) of a random subtree.

    Start from the root of the full depth x width tree and grow an
    ancestor-closed node set by adding a uniformly chosen frontier node until
    n_nodes nodes are present.  Nodes are then numbered in BFS order with
    siblings in the order of their slot in the full tree.
    """
    full = sum(width ** d for d in range(depth + 1))
    if not 1 <= n_nodes <= full:
        raise ValueError("n_nodes outside [1, full tree size]")
    chosen = {()}
    frontier = [(c,) for c in range(width)] if depth > 0 else []
    while len(chosen) < n_nodes:
        i = int(rng.integers(len(frontier)))
        node = frontier.pop(i)
        chosen.add(node)
        if len(node) < depth:
            frontier.extend(node + (c,) for c in range(width))
    order = sorted(chosen, key=lambda p: (len(p), p))
    index = {p: i for i, p in enumerate(order)}
    parent = np.full(n_nodes, -1, dtype=np.int32)
    for p, i in index.items():
        if p:
            parent[i] = index[p[:-1]]
    return parent


def _gumbel_argmax(rng: np.random.Generator, scaled_logits: np.ndarray) -> int:
    g = -np.log(-np.log(rng.random(scaled_logits.shape[-1])))
    return int(np.argmax(scaled_logits + g))


# ---------------------------------------------------------------------------
# logits / tokens / tree
# ---------------------------------------------------------------------------

def logits_inputs(wl: Workload, seed: int, B: int | None = None) -> dict:
    """Target/draft logits, draft tokens, tree topology and temperatures.

    Returns a dict of numpy arrays:
      target, draft : [B, M, V] float32 (bf16-exact for bf16 workloads)
      tokens        : [B, M] int32; tokens[b, 0] is the pending root token
      parent        : [B, M] int32 (tree) or None (chain)
      temperature   : [B] float32
    Row n of target/draft is the distribution over the children of node n.
    The token of node c is drawn from softmax(draft[b, parent(c)] / T).
    """
    B = wl.B if B is None else B
    M, V = wl.M, wl.V
    rng = np.random.default_rng([seed, 1])
    target = np.empty((B, M, V), dtype=np.float32)
    draft = np.empty((B, M, V), dtype=np.float32)
    for b in range(B):
        z = rng.standard_normal((M, V), dtype=np.float32) * np.float32(wl.sigma)
        z = _cast(z, wl.dtype)
        n = rng.standard_normal((M, V), dtype=np.float32) * np.float32(wl.noise)
        target[b] = z
        draft[b] = _cast(z + n, wl.dtype)
    parent = None
    if wl.is_tree:
        parent = np.stack([random_tree(rng, wl.gamma, wl.tree_width, M)
                           for _ in range(B)]).astype(np.int32)
    tokens = np.empty((B, M), dtype=np.int32)
    for b in range(B):
        tokens[b, 0] = int(rng.integers(V))
        for c in range(1, M):
            par = c - 1 if parent is None else int(parent[b, c])
            row = draft[b, par].astype(np.float64) / wl.T
            tokens[b, c] = _gumbel_argmax(rng, row)
    temperature = np.full(B, wl.T, dtype=np.float32)
    return dict(target=target, draft=draft, tokens=tokens, parent=parent,
                temperature=temperature)


# ---------------------------------------------------------------------------
# paged KV cache
# ---------------------------------------------------------------------------

def kv_layout(wl: Workload, seed: int, B: int | None = None,
              ctx: np.ndarray | None = None, slack_blocks: int = 3) -> dict:
    """Context lengths and block tables (a random permutation of blocks).

    Request b owns ceil((ctx_b + M) / block) blocks; table entries past that
    are -1.  A few spare physical blocks are never referenced.
    """
    B = wl.B if B is None else B
    if ctx is None:
        ctx = context_lengths(wl, seed)[:B]
    ctx = np.asarray(ctx, dtype=np.int32)
    need = (ctx.astype(np.int64) + wl.M + wl.block - 1) // wl.block
    max_blocks = int(need.max())
    num_blocks = int(need.sum()) + slack_blocks
    rng = np.random.default_rng([seed, 3])
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, :need[b]] = perm[off:off + need[b]]
        off += int(need[b])
    return dict(ctx_lens=ctx, block_table=table, num_blocks=num_blocks,
                max_blocks=max_blocks)


def kv_inputs_host(wl: Workload, seed: int, B: int | None = None,
                   ctx: np.ndarray | None = None) -> dict:
    """Queries, new K/V and a full paged cache generated on the host.

    Arrays are float32 holding bf16-exact values for bf16 workloads.
    Shapes: q [B, M, Hq, D]; k_new, v_new [B, M, Hkv, D];
    k_cache, v_cache [num_blocks, Hkv, block, D].
    """
    lay = kv_layout(wl, seed, B=B, ctx=ctx)
    B = lay["block_table"].shape[0]
    rng = np.random.default_rng([seed, 4])
    M, Hq, Hkv, D = wl.M, wl.Hq, wl.Hkv, wl.D

    def normal(*shape):
        return _cast(rng.standard_normal(shape, dtype=np.float32), wl.dtype)

    q = normal(B, M, Hq, D)
    k_new = normal(B, M, Hkv, D)
    v_new = normal(B, M, Hkv, D)
    k_cache = normal(lay["num_blocks"], Hkv, wl.block, D)
    v_cache = normal(lay["num_blocks"], Hkv, wl.block, D)
    out = dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache,
               v_cache=v_cache)
    out.update(lay)
    return out


def kv_cache_bytes(wl: Workload, num_blocks: int) -> int:
    esize = 2 if wl.dtype == "bf16" else 4
    return 2 * num_blocks * wl.Hkv * wl.block * wl.D * esize


def expected_ctx_mean(wl: Workload) -> float:
    if wl.ctx[0] == "fixed":
        return float(wl.ctx[1])
    return 0.5 * (wl.ctx[1] + wl.ctx[2])


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)



def kv_inputs_device(wl: Workload, seed: int, device, B: int | None = None,
                     ctx: np.ndarray | None = None) -> dict:
    """Like kv_inputs_host, but the large caches are drawn on the device.

    Block tables, context lengths, queries and the new K/V rows come from the
    host generator (same values as kv_inputs_host); the two caches are drawn
    with torch's seeded device generator, so full-size workloads (several GB
    of cache) need no host round trip.  Returns torch tensors on `device`
    (bf16 or fp32) plus the layout arrays as numpy.
    """
    import torch

    lay = kv_layout(wl, seed, B=B, ctx=ctx)
    Bn = lay["block_table"].shape[0]
    rng = np.random.default_rng([seed, 4])
    M, Hq, Hkv, D = wl.M, wl.Hq, wl.Hkv, wl.D

    def normal(*shape):
        return _cast(rng.standard_normal(shape, dtype=np.float32), wl.dtype)

    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    q = torch.from_numpy(normal(Bn, M, Hq, D)).to(device=device, dtype=tdt)
    k_new = torch.from_numpy(normal(Bn, M, Hkv, D)).to(device=device, dtype=tdt)
    v_new = torch.from_numpy(normal(Bn, M, Hkv, D)).to(device=device, dtype=tdt)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    shape = (lay["num_blocks"], Hkv, wl.block, D)
    k_cache = torch.randn(shape, generator=g, device=device, dtype=tdt)
    v_cache = torch.randn(shape, generator=g, device=device, dtype=tdt)
    out = dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache)
    out.update(lay)
    return out
