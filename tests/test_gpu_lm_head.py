"""GPU parity of the LM head (spec_lm_head) and of the LM heads fused with the
verify decisions (spec_reject_sample_lm_head) against the CPU oracle.

* logits: the GPU's bf16 output (fp32 accumulation on the tensor cores) is
  the fp64 product rounded to bf16, within one bf16 step plus the fp32
  accumulation error;
* decisions: the fused call's accepted lengths, paths and tokens are those
  of the oracle run on the logits the fused call wrote (bit-exact outside
  the near-threshold bands), and its probe (whose p(x), q(x) come from the
  statistics the LM heads formed in their epilogue) within 1e-5 -- so the
  epilogue's statistics equal what the statistics pass would find;
* ragged row counts, vocabularies that end inside a statistics chunk, a
  tree, temperature-0 requests, and the shapes the kernel refuses.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import compare_reject  # noqa: E402
from oracle import oracle_lm_head, oracle_reject_sample  # noqa: E402
from synth import bf16_round, random_tree  # noqa: E402


def _bf16(rng, shape, scale):
    return bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))


def _dev(x, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dt)


def _check_logits(g, z):
    # one bf16 step of the value (2^-8 relative) plus the accumulation error
    err = np.abs(g.astype(np.float64) - z)
    tol = np.abs(z) * 2.0 ** -8 + 2e-3
    assert np.all(err <= tol), float((err - tol).max())


@pytest.mark.parametrize("rows,H,V", [(128, 64, 256), (300, 256, 2304), (640, 1024, 8192)])
def test_lm_head_matches_oracle(rows, H, V):
    rng = np.random.default_rng(rows + H)
    h = _bf16(rng, (rows, H), 1.0)
    w = _bf16(rng, (V, H), 3.0 / np.sqrt(H))
    logits = torch.full((rows, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    launches = sv.spec_lm_head(_dev(h), _dev(w), logits, ws)
    torch.cuda.synchronize()
    assert launches == 1
    _check_logits(logits.float().cpu().numpy(), oracle_lm_head(h, w))


def test_lm_head_refuses_unsupported_shapes():
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    for H, V in [(100, 256), (64, 300)]:
        h = torch.zeros(4, H, dtype=torch.bfloat16, device="cuda")
        w = torch.zeros(V, H, dtype=torch.bfloat16, device="cuda")
        out = torch.zeros(4, V, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(sv.SpecError) as e:
            sv.spec_lm_head(h, w, out, ws)
        assert e.value.code == 3


def _fused(B, gamma, V, Ht, Hd, T, seed, tree=None, offset=0):
    rng = np.random.default_rng(seed)
    M = gamma + 1 if tree is None else len(tree)
    ht = _bf16(rng, (B, M, Ht), 1.0)
    wt = _bf16(rng, (V, Ht), 3.0 / np.sqrt(Ht))
    # the draft head sees a noisy copy of the target's hidden state through
    # a smaller hidden size: its logits track the target's loosely
    hd = _bf16(rng, (B, M, Hd), 1.0)
    wd = _bf16(rng, (V, Hd), 3.0 / np.sqrt(Hd))
    zt = oracle_lm_head(ht, wt)
    zd = oracle_lm_head(hd, wd)
    parent = None if tree is None else np.tile(np.asarray(tree, np.int32), (B, 1))
    tokens = np.zeros((B, M), np.int32)
    for b in range(B):
        for c in range(1, M):
            pn = c - 1 if parent is None else parent[b, c]
            # half of the drafts are the target's argmax, so that acceptances happen
            tokens[b, c] = int(np.argmax(zt[b, pn])) if (b + c) % 2 else int(rng.integers(V))
    temp = np.full(B, T, np.float32)
    temp[::3] = 0.0  # some greedy requests in the same call
    dims = sv.make_dims(B=B, M=M, V=V, logits_dtype=torch.bfloat16)
    ws = sv.workspace(dims)
    tl = torch.full((B, M, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    dl = torch.full_like(tl, float("nan"))
    out = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, M), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    pr = torch.full((B, M, 4), float("nan"), dtype=torch.float32, device="cuda")
    sv.spec_reject_sample_lm_head(_dev(ht), _dev(wt), _dev(hd), _dev(wd), tl, dl, _dev(tokens, torch.int32),
                                  None if parent is None else _dev(parent, torch.int32),
                                  _dev(temp, torch.float32), 11, offset, out, path, acc, pr,
                                  dims, ws)
    torch.cuda.synchronize()
    g = dict(out_tokens=out.cpu().numpy(), path=path.cpu().numpy(),
             accepted_len=acc.cpu().numpy(), probe=pr.cpu().numpy(), status=sv.device_status(ws))
    gt, gd = tl.float().cpu().numpy(), dl.float().cpu().numpy()
    _check_logits(gt, zt)
    _check_logits(gd, zd)
    o = oracle_reject_sample(gt, gd, tokens, parent, temp, 11, offset)
    return g, o


@pytest.mark.parametrize("B,gamma,V,Ht,Hd", [(8, 5, 8192, 512, 256), (5, 3, 2304, 256, 128),
                                            (3, 8, 33024, 1024, 512)])
def test_fused_chain_matches_oracle(B, gamma, V, Ht, Hd):
    for offset in range(2):
        g, o = _fused(B, gamma, V, Ht, Hd, 0.9, seed=B * 10 + gamma, offset=offset)
        assert g["status"] == 0
        near = compare_reject(g, o)
        assert near <= 1
    assert (o["accepted_len"] > 0).any()


def test_fused_tree_matches_oracle():
    tree = random_tree(np.random.default_rng(5), 3, 3, 16)
    g, o = _fused(4, 3, 4096, 256, 128, 1.0, seed=9, tree=tree)
    assert g["status"] == 0
    compare_reject(g, o)
