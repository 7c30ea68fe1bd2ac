"""Paged-KV append and verify attention, fp64 on the CPU.

The target model scores all g + 1 new positions (the pending root token and
the g drafts), or every node of a draft tree, in one forward pass.  Under the
causal mask each position sees only what precedes it, so the parallel pass
equals token-by-token decoding (page 1 §2.1; page 2 §2.1 and §3.3: the cached
prefix is reused and only the new positions get fresh K/V).  For a draft tree
each node sees the cached prefix, its ancestors and itself (page 3,
tree-attention section: the verify pass must follow the tree's shape as its
mask; page 2 §5.4: the mask matrix of a batched tree verify).

Readings taken where the pages are silent:
* keys and queries arrive with any position encoding already applied;
* scores are scaled by 1/sqrt(D) unless a scale is given;
* grouped-query attention: query head h reads KV head h // (Hq / Hkv);
* the paged cache is [num_blocks, Hkv, block, D]; position t of request b
  lives in block block_table[b, t // block], slot t % block (the pages speak
  of a PagedAttention block table, page 2 §4.3 and page 3);
* the append writes the new K/V of the M new rows at positions
  ctx .. ctx + M - 1 and clears the rest of the last block it touches, so
  stale or uninitialised bytes never sit inside a block that is read.
"""
from __future__ import annotations

import numpy as np


def ancestors_or_self(parent: np.ndarray | None, i: int) -> list:
    """Node indices from the root to node i (inclusive); chain if parent is None."""
    if parent is None:
        return list(range(i + 1))
    chain = []
    n = i
    while n >= 0:
        chain.append(n)
        n = int(parent[n])
    return chain[::-1]


def gather_positions(cache: np.ndarray, table_row: np.ndarray,
                     positions: np.ndarray, block: int) -> np.ndarray:
    """cache[block_of(t), :, slot_of(t), :] for each position t -> [n, Hkv, D]."""
    positions = np.asarray(positions, dtype=np.int64)
    blk = table_row[positions // block]
    slot = positions % block
    return cache[blk, :, slot, :]


def oracle_kv_append(k_cache, v_cache, block_table, ctx_lens, k_new, v_new,
                     block=16):
    """Caches after writing each request's M new K/V rows (copies returned)."""
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    B, M = k_new.shape[:2]
    for b in range(B):
        ctx = int(ctx_lens[b])
        for i in range(M):
            t = ctx + i
            blk = block_table[b, t // block]
            k[blk, :, t % block, :] = k_new[b, i]
            v[blk, :, t % block, :] = v_new[b, i]
        end = -(-(ctx + M) // block) * block
        for t in range(ctx + M, end):
            blk = block_table[b, t // block]
            k[blk, :, t % block, :] = 0
            v[blk, :, t % block, :] = 0
    return k, v


def oracle_verify_attn(q, k_cache, v_cache, block_table, ctx_lens, k_new,
                       v_new, parent=None, scale=None, block=16):
    """Batched masked verify attention after the append.

    q [B, M, Hq, D]; caches [num_blocks, Hkv, block, D] (before the append);
    k_new, v_new [B, M, Hkv, D]; parent [B, M] or None (chain).
    Returns (out [B, M, Hq, D] fp64, lse [B, M, Hq] fp64 natural-log
    log-sum-exp of the scaled scores, k_after, v_after).
    """
    q = np.asarray(q, dtype=np.float64)
    B, M, Hq, D = q.shape
    Hkv = k_new.shape[2]
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kc, vc = oracle_kv_append(k_cache, v_cache, block_table, ctx_lens, k_new,
                              v_new, block)
    out = np.zeros((B, M, Hq, D), dtype=np.float64)
    lse = np.zeros((B, M, Hq), dtype=np.float64)
    for b in range(B):
        ctx = int(ctx_lens[b])
        L = ctx + M
        pos = np.arange(L)
        K = gather_positions(kc, block_table[b], pos, block).astype(np.float64)
        V = gather_positions(vc, block_table[b], pos, block).astype(np.float64)
        par = None if parent is None else np.asarray(parent[b])
        visible = np.zeros((M, L), dtype=bool)
        visible[:, :ctx] = True
        for i in range(M):
            for a in ancestors_or_self(par, i):
                visible[i, ctx + a] = True
        for h in range(Hq):
            g = h // group
            s = (q[b, :, h, :] @ K[:, g, :].T) * scale          # [M, L]
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            w = np.exp(s - m)
            lsum = w.sum(axis=1, keepdims=True)
            out[b, :, h, :] = (w @ V[:, g, :]) / lsum
            lse[b, :, h] = (m + np.log(lsum))[:, 0]
    return out, lse, kc, vc


def oracle_verify_attn_tokenwise(q, k_cache, v_cache, block_table, ctx_lens,
                                 k_new, v_new, parent=None, scale=None,
                                 block=16):
    """The same outputs by decoding one position at a time.

    For every node i, its keys are the cached prefix followed by the new K/V
    of its ancestors in root-to-node order (for a chain: the previous new
    positions), exactly what token-by-token decoding would have cached before
    scoring position i.  No mask is formed.
    """
    q = np.asarray(q, dtype=np.float64)
    B, M, Hq, D = q.shape
    Hkv = k_new.shape[2]
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, M, Hq, D), dtype=np.float64)
    lse = np.zeros((B, M, Hq), dtype=np.float64)
    for b in range(B):
        ctx = int(ctx_lens[b])
        Kp = gather_positions(k_cache, block_table[b], np.arange(ctx), block)
        Vp = gather_positions(v_cache, block_table[b], np.arange(ctx), block)
        par = None if parent is None else np.asarray(parent[b])
        for i in range(M):
            chain = ancestors_or_self(par, i)
            K = np.concatenate([Kp, k_new[b, chain]]).astype(np.float64)
            V = np.concatenate([Vp, v_new[b, chain]]).astype(np.float64)
            for h in range(Hq):
                g = h // group
                s = (K[:, g, :] @ q[b, i, h, :]) * scale
                m = s.max()
                w = np.exp(s - m)
                out[b, i, h, :] = (w @ V[:, g, :]) / w.sum()
                lse[b, i, h] = m + np.log(w.sum())
    return out, lse
