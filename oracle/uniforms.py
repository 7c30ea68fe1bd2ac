"""Counter-based uniforms for the accept tests and the resample draws.

The pages only say the draws are random (page 1 §4.3 insists on keeping the
sampling random).  The reading adopted here: each decision takes its uniform
from Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
easy as 1, 2, 3", SC'11), so that any implementation can reproduce the draws
without sharing state.

For request b (plus a caller-chosen request base), node n and call offset o:
    key      = (seed, 0)
    counter  = (n + 1, b_base + b, o, 0)
    w0..w3   = Philox4x64-10(counter, key)
    u_acc(n) = (w0 >> 40) * 2^-24      uniform of the accept test of node n
    u_smp(n) = (w1 >> 40) * 2^-24      uniform of a sample drawn at node n
Both lie in [0, 1) on a 2^-24 grid, so they are exact in fp32 and fp64.

numpy's Philox bit generator is Philox4x64-10 and advances its counter by one
before producing a block, so seeding it with counter (n, b, o, 0) yields the
block of counter (n + 1, b, o, 0).
"""
from __future__ import annotations

import numpy as np

_TWO_M24 = 2.0 ** -24


def _u64(words):
    # numpy routes plain Python-int lists through float64, which corrupts
    # words above 2^53; pass explicit uint64 arrays.
    return np.array([int(w) % (1 << 64) for w in words], dtype=np.uint64)


def philox_block(seed: int, counter: tuple) -> np.ndarray:
    """The four 64-bit words of Philox4x64-10 at `counter` under key (seed, 0).

    `counter` must have a nonzero first word (it is decremented by one to
    account for numpy's pre-increment).
    """
    c0, c1, c2, c3 = (int(x) for x in counter)
    if c0 == 0:
        raise ValueError("first counter word must be >= 1")
    g = np.random.Philox(key=_u64([seed, 0]), counter=_u64([c0 - 1, c1, c2, c3]))
    return g.random_raw(4).astype(np.uint64)


def uniforms_for(seed: int, offset: int, b_global: int, n_nodes: int):
    """(u_acc[n_nodes], u_smp[n_nodes]) of one request."""
    # Counters (1, b, o, 0) .. (n_nodes, b, o, 0) differ only in word 0, so
    # one generator started at (0, b, o, 0) yields their blocks in order.
    g = np.random.Philox(key=_u64([seed, 0]),
                         counter=_u64([0, b_global, offset, 0]))
    w = g.random_raw(4 * n_nodes).astype(np.uint64).reshape(n_nodes, 4)
    u_acc = (w[:, 0] >> np.uint64(40)).astype(np.float64) * _TWO_M24
    u_smp = (w[:, 1] >> np.uint64(40)).astype(np.float64) * _TWO_M24
    return u_acc, u_smp
