"""Helpers shared by the GPU parity tests: upload seeded inputs, call the
library through its C ABI binding, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import speculative_decoding_verification_19_gb300 as sv
from oracle import (FILTER_NEAR, oracle_kv_append, oracle_kv_commit, oracle_reject_sample,
                    oracle_verify_attn)

ATT_ABS, ATT_REL = 2e-2, 1e-2      # attention outputs (bf16 in, fp32 accumulate)
LSE_ABS = 1e-3                     # log-sum-exp (fp32)
PROB_ABS = 1e-5                    # probabilities in the probe
NEAR = 1e-6                        # near-threshold draws are excluded


def tdtype(wl):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def to_dev(x, dt, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=dev, dtype=dt)


def dims_for(wl, B, max_blocks=1, num_blocks=1, V=None, impl=0):
    return sv.make_dims(B=B, M=wl.M, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D,
                        max_blocks=max_blocks, num_blocks=num_blocks,
                        V=wl.V if V is None else V, kv_dtype=tdtype(wl),
                        logits_dtype=tdtype(wl), attn_impl=impl)


def impls_for(wl):
    """Attention kernels that support this shape (CUDA cores, tensor cores)."""
    R = (wl.Hq // wl.Hkv) * wl.M
    out = []
    if R <= 128:
        out.append(sv.ATTN_CUDA_CORES)
    if wl.dtype == "bf16" and wl.D == 128 and R <= 128:
        out.append(sv.ATTN_TENSOR_CORES)
    return out


# ---------------------------------------------------------------------------
# reject sample
# ---------------------------------------------------------------------------

def gpu_reject(wl, lg, seed, offset, b_base=0, dims=None, ws=None, probe=True, top_k=None,
               top_p=None):
    B, M, V = lg["target"].shape
    dt = tdtype(wl)
    dims = dims or dims_for(wl, B, V=V)
    ws = sv.workspace(dims) if ws is None else ws
    t = to_dev(lg["target"], dt)
    d = to_dev(lg["draft"], dt)
    tok = to_dev(lg["tokens"], torch.int32)
    par = None if lg["parent"] is None else to_dev(lg["parent"], torch.int32)
    temp = to_dev(lg["temperature"], torch.float32)
    # sentinel-filled: anything the kernels leave unwritten fails the comparison
    out_tokens = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    pr = torch.full((B, M, 4), float("nan"), dtype=torch.float32, device="cuda") if probe else None
    tk = None if top_k is None else to_dev(top_k, torch.int32)
    tp = None if top_p is None else to_dev(top_p, torch.float32)
    sv.spec_reject_sample(t, d, tok, par, temp, seed, offset, out_tokens, path,
                          acc, pr, dims, ws, b_base=b_base, top_k=tk, top_p=tp)
    torch.cuda.synchronize()
    res = dict(out_tokens=out_tokens.cpu().numpy(), path=path.cpu().numpy(),
               accepted_len=acc.cpu().numpy(),
               status=sv.device_status(ws))
    if probe:
        res["probe"] = pr.cpu().numpy()
    return res


def compare_reject(g, o):
    """Parity of the verify decisions.

    Requests whose accept tests are all clear of their thresholds by 1e-6
    must match bit-exactly in accepted length, path and accepted tokens.  The
    final draw must match exactly too when it is clear of its CDF steps;
    otherwise the GPU's token must lie in the oracle's band (the tokens a
    draw within 1e-6 of u could select) and carry positive mass.  Returns
    the number of requests with a near-threshold accept test (excluded).
    A request whose top-p cut lies within FILTER_NEAR (relative) of its
    target mass is excluded the same way (its kept set is ambiguous).
    """
    bad = o["status"] != 0
    assert np.array_equal(g["accepted_len"][bad], o["accepted_len"][bad])
    acc_clear = (o["acc_margin"] >= NEAR) & ~bad
    if "flt_margin" in o:
        acc_clear &= o["flt_margin"] >= FILTER_NEAR
    for key in ("accepted_len", "path"):
        assert np.array_equal(g[key][acc_clear], o[key][acc_clear]), key
    B, M = o["path"].shape
    for b in np.nonzero(acc_clear)[0]:
        a = o["accepted_len"][b]
        assert np.array_equal(g["out_tokens"][b, :a], o["out_tokens"][b, :a])
        assert np.all(g["out_tokens"][b, a + 1:] == -1)
        if o["smp_margin"][b] >= NEAR:
            assert g["out_tokens"][b, a] == o["out_tokens"][b, a]
        else:
            lo, hi = o["band"][b]
            assert lo <= g["out_tokens"][b, a] <= hi, (b, lo, hi)
    if "probe" in g:
        sel = acc_clear
        gp, op = g["probe"][sel], o["probe"][sel]
        unset = op == -1.0
        assert np.array_equal(gp[unset], op[unset])
        # the probability of the drawn token is compared only where the
        # draw itself is clear of its thresholds
        clear_draw = (o["smp_margin"][sel] >= NEAR)[:, None]
        cmp = ~unset.copy()
        cmp[:, :, 3] &= np.broadcast_to(clear_draw, cmp[:, :, 3].shape)
        assert np.max(np.abs(gp[cmp] - op[cmp]), initial=0.0) <= PROB_ABS
    return int((~acc_clear & ~bad).sum())


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def gpu_attn(wl, kv, parent=None, dims=None, ws=None, impl=0):
    """kv: host dict from synth.kv_inputs_host.  Returns numpy outputs."""
    dt = tdtype(wl)
    B = kv["block_table"].shape[0]
    dims = dims or dims_for(wl, B, kv["max_blocks"], kv["num_blocks"], impl=impl)
    ws = sv.workspace(dims) if ws is None else ws
    q = to_dev(kv["q"], dt)
    kn = to_dev(kv["k_new"], dt)
    vn = to_dev(kv["v_new"], dt)
    kc = to_dev(kv["k_cache"], dt)
    vc = to_dev(kv["v_cache"], dt)
    bt = to_dev(kv["block_table"], torch.int32)
    ctx = to_dev(kv["ctx_lens"], torch.int32)
    par = None if parent is None else to_dev(parent, torch.int32)
    # NaN-filled: an output row the kernels never write fails the comparison
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    sv.spec_verify_attn(q, kn, vn, kc, vc, bt, ctx, par, out, lse, dims, ws)
    torch.cuda.synchronize()
    return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy(),
                k_cache=kc.float().cpu().numpy(), v_cache=vc.float().cpu().numpy(),
                status=sv.device_status(ws), dev=dict(kc=kc, vc=vc, bt=bt, ctx=ctx,
                                                       dims=dims, ws=ws))


def oracle_attn(wl, kv, parent=None):
    return oracle_verify_attn(kv["q"], kv["k_cache"], kv["v_cache"],
                              kv["block_table"], kv["ctx_lens"], kv["k_new"],
                              kv["v_new"], parent=parent, block=wl.block)


def assert_attn_close(g_out, o_out, g_lse=None, o_lse=None):
    err = np.abs(g_out - o_out)
    tol = ATT_ABS + ATT_REL * np.abs(o_out)
    assert np.all(err <= tol), f"max err {err.max():.3e}"
    if g_lse is not None:
        assert np.max(np.abs(g_lse - o_lse)) <= LSE_ABS


def cache_equal_except(a, b, block_table, lo, hi, block=16):
    """a == b bit-exactly except positions [lo_b, hi_b) of each request."""
    a = a.copy()
    b = b.copy()
    for r in range(len(lo)):
        for t in range(int(lo[r]), int(hi[r])):
            blk = block_table[r, t // block]
            a[blk, :, t % block] = 0
            b[blk, :, t % block] = 0
    return np.array_equal(a, b)


__all__ = [n for n in dir() if not n.startswith("_")] + [
    "oracle_kv_append", "oracle_kv_commit", "oracle_reject_sample"]
