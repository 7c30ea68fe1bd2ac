"""GPU parity of spec_reject_sample_filtered (top-k / top-p restricted laws)
against the CPU oracle.

Each request carries its own filter (none, top-k, top-p or both, mixed in
one call); the accepted lengths, paths and tokens are bit-exact outside the
near-threshold bands, the probe (the restricted laws' probabilities) within
1e-5.  Covers full-size chain and tree workloads, bf16 rows full of equal
logits (ties at the cut), unaligned fp32 rows, k = 1 against greedy decoding,
invalid filters and the refusal of the one-kernel path.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import compare_reject, dims_for, gpu_reject  # noqa: E402
from oracle import oracle_reject_sample  # noqa: E402
from synth import logits_inputs, workload  # noqa: E402


def _filters(B, V, seed):
    """A mix of per-request filters: none, top-k, top-p, both."""
    rng = np.random.default_rng(seed)
    k = np.zeros(B, np.int32)
    p = np.ones(B, np.float32)
    for b in range(B):
        kind = b % 4
        if kind in (1, 3):
            k[b] = int(rng.choice([1, 2, 20, 1000, V - 1]))
        if kind in (2, 3):
            p[b] = float(rng.choice([0.3, 0.5, 0.9, 0.95, 0.999]))
    return k, p


def _run(wl, lg, seed, offset, top_k, top_p, impl=sv.REJECT_AUTO):
    B, M, V = lg["target"].shape
    dims = dims_for(wl, B, V=V)
    dims.reject_impl = impl
    g = gpu_reject(wl, lg, seed, offset, dims=dims, top_k=top_k, top_p=top_p)
    o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], lg["parent"],
                             lg["temperature"], seed, offset, top_k=top_k, top_p=top_p)
    near = compare_reject(g, o)
    return g, o, near


@pytest.mark.parametrize("name,B", [("chain_gqa_128k", 32), ("chain_7b", 8),
                                    ("tree_64", 6)])
def test_filtered_workloads(name, B):
    wl = workload(name)
    lg = logits_inputs(wl, seed=17, B=B)
    V = wl.V
    k, p = _filters(B, V, seed=3)
    for offset in range(2):
        g, o, near = _run(wl, lg, 5, offset, k, p)
        assert g["status"] == 0
        assert near <= max(1, B // 8)
    # the filters change the outcome of some requests
    u = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], lg["parent"],
                             lg["temperature"], 5, 1)
    assert not np.array_equal(u["out_tokens"], o["out_tokens"])


def test_ties_at_the_cut():
    # integer-valued logits: hundreds of equal values, so every cut falls
    # inside a group of ties and the smaller indices decide
    wl = workload("chain_7b").scaled(B=8, V=3000, gamma=3)
    lg = logits_inputs(wl, seed=18)
    rng = np.random.default_rng(4)
    for key in ("target", "draft"):
        lg[key] = np.round(lg[key]).astype(np.float32)
    k = np.array([5, 50, 0, 0, 7, 300, 1, 0], np.int32)
    p = np.array([1.0, 1.0, 0.5, 0.9, 0.6, 0.8, 1.0, 0.97], np.float32)
    del rng
    for offset in range(3):
        g, o, near = _run(wl, lg, 6, offset, k, p)
        assert g["status"] == 0


@pytest.mark.parametrize("V", [300, 4099])
def test_unaligned_fp32_rows(V):
    wl = workload("chain_7b").scaled(B=6, V=V, dtype="f32", gamma=4)
    lg = logits_inputs(wl, seed=19)
    k, p = _filters(6, V, seed=5)
    for offset in range(2):
        _run(wl, lg, 7, offset, k, p)


def test_top_k_one_is_greedy_on_the_gpu():
    wl = workload("chain_7b").scaled(B=8, V=5000)
    lg = logits_inputs(wl, seed=20)
    t = lg["target"]
    for b in range(wl.B):
        for c in range(1, wl.M):
            if (b + c) % 2:
                lg["tokens"][b, c] = int(np.argmax(t[b, c - 1]))
    g1, _, _ = _run(wl, lg, 8, 0, np.ones(wl.B, np.int32), None)
    greedy = dict(lg, temperature=np.zeros(wl.B, np.float32))
    g0 = gpu_reject(wl, greedy, 8, 0)
    for key in ("out_tokens", "path", "accepted_len"):
        assert np.array_equal(g1[key], g0[key])
    assert (g1["accepted_len"] > 0).any()


def test_invalid_filters_fail_their_requests():
    wl = workload("chain_7b").scaled(B=5, V=4096)
    lg = logits_inputs(wl, seed=21)
    k = np.array([0, -1, 0, 0, 3], np.int32)
    p = np.array([0.9, 1.0, 0.0, 1.5, np.nan], np.float32)
    g, o, _ = _run(wl, lg, 9, 0, k, p)
    assert list(g["accepted_len"][1:]) == [-1, -1, -1, -1]
    assert g["accepted_len"][0] >= 0
    assert g["status"] == (1 << 1)  # SPEC_ERR_INVALID_ARG


def test_one_kernel_path_refuses_filters():
    wl = workload("chain_7b").scaled(B=2, V=4096)
    lg = logits_inputs(wl, seed=22)
    dims = dims_for(wl, 2, V=4096)
    dims.reject_impl = sv.REJECT_FUSED
    with pytest.raises(sv.SpecError) as e:
        gpu_reject(wl, lg, 1, 0, dims=dims, top_k=np.array([3, 3], np.int32))
    assert e.value.code == 3
