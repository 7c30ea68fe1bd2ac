"""KV commit after the verify decisions, on the CPU.

Page 2 §3.3: the verify pass caches K/V for every draft position; when the
drafts are rejected from position i on, the cache from i on is dropped and the
sequence rolls back to the accepted prefix.  Page 2 §5.4 and page 3 (tree
section) add that a tree verify must roll back along a dynamic path.

Readings taken:
* the K/V of the root and of the a accepted nodes are kept; the replacement /
  bonus token sampled this step has no K/V yet (it is the next step's root),
  so the new context length is ctx + a + 1;
* for a chain the kept rows already sit at ctx .. ctx + a, so the commit is a
  length update;
* for a tree, row j of the accepted path (node path[j]) is moved from slot
  ctx + path[j] to slot ctx + j, for j = 1 .. a in increasing order; slots from
  the new length on are left as they are (they are free);
* a failed request (accepted length -1) keeps its length and its cache.
"""
from __future__ import annotations

import numpy as np


def oracle_kv_commit(k_cache, v_cache, block_table, ctx_lens, path,
                     accepted_len, block=16):
    """Returns (k_after, v_after, new_ctx_lens); inputs are not modified."""
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    new_ctx = np.array(ctx_lens, dtype=np.int32, copy=True)
    B = len(ctx_lens)
    for b in range(B):
        a = int(accepted_len[b])
        if a < 0:
            continue
        ctx = int(ctx_lens[b])
        for j in range(1, a + 1):
            src = ctx + int(path[b, j])
            dst = ctx + j
            if src == dst:
                continue
            sb, ss = block_table[b, src // block], src % block
            db, ds = block_table[b, dst // block], dst % block
            k[db, :, ds, :] = k[sb, :, ss, :]
            v[db, :, ds, :] = v[sb, :, ss, :]
        new_ctx[b] = ctx + a + 1
    return k, v, new_ctx
