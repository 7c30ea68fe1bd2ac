"""GPU parity of spec_reject_sample against the CPU oracle.

Bit-exact accepted lengths, paths and emitted tokens for every request whose
draws are clear of their thresholds by 1e-6 (the oracle reports the margin);
probe probabilities within 1e-5.  Covers the five workloads at their full
batch and vocabulary, ragged and unaligned vocabularies, trees, the
all-accept / all-reject edge cases, failed requests, and a 10^6-trial
chi-square of the GPU's own output law.
"""
import numpy as np
import pytest
import torch
from scipy import stats

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import compare_reject, dims_for, gpu_reject  # noqa: E402
from oracle import oracle_reject_sample, softmax_rows  # noqa: E402
from synth import bf16_round, logits_inputs, workload  # noqa: E402


IMPLS = [sv.REJECT_FUSED, sv.REJECT_STAGED]
# trees run on the staged kernels; the one-kernel path takes chains only
TREE_IMPLS = [sv.REJECT_AUTO, sv.REJECT_STAGED]


def _aligned(wl, V):
    return (V * (2 if wl.dtype == "bf16" else 4)) % 16 == 0


def _run(wl, lg, seed, offset, b_base=0, impl=sv.REJECT_AUTO):
    B, M, V = lg["target"].shape
    dims = dims_for(wl, B, V=V)
    dims.reject_impl = impl
    if impl == sv.REJECT_FUSED and (lg["parent"] is not None or not _aligned(wl, V)):
        with pytest.raises(sv.SpecError) as err:
            gpu_reject(wl, lg, seed, offset, b_base=b_base, dims=dims)
        assert err.value.code == 3  # SPEC_ERR_UNSUPPORTED: nothing launched
        dims.reject_impl = sv.REJECT_AUTO
    g = gpu_reject(wl, lg, seed, offset, b_base=b_base, dims=dims)
    o = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"],
                             lg["parent"], lg["temperature"], seed, offset,
                             b_base=b_base)
    near = compare_reject(g, o)
    return g, o, near


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["tiny_chain", "chain_7b", "chain_gqa_128k",
                                  "tree_64", "stress_gqa_152k"])
def test_workload_full_size(name, impl):
    wl = workload(name)
    lg = logits_inputs(wl, seed=0)
    total_near = 0
    for offset in (0, 1, 2):
        g, o, near = _run(wl, lg, seed=1234, offset=offset, impl=impl)
        total_near += near
        assert g["status"] == 0
    # near-threshold exclusions must stay rare
    assert total_near <= max(1, wl.B // 20)


@pytest.mark.parametrize("B,gamma,V", [(1, 1, 8), (3, 2, 32), (3, 8, 1000),
                                       (2, 5, 32007), (4, 3, 4097), (2, 8, 50),
                                       (3, 0, 4096)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("impl", [sv.REJECT_FUSED, sv.REJECT_STAGED])
def test_ragged_shapes(B, gamma, V, dtype, impl):
    # the staged path: the chain tail kernel where the rows are 16-byte
    # aligned (V a multiple of 8 for bf16, of 4 for fp32), the scalar
    # kernels elsewhere; the one-kernel path refuses unaligned rows
    wl = workload("chain_7b").scaled(B=B, gamma=gamma, V=V, dtype=dtype, T=0.9)
    lg = logits_inputs(wl, seed=B * 100 + gamma)
    for offset in range(3):
        _run(wl, lg, seed=99, offset=offset, b_base=5, impl=impl)


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (2, 63, 1000, "bf16"),      # the longest chain: M = 64 rows
    (2, 3, 1 << 20, "bf16"),    # the largest vocabulary: 512 statistics chunks per row
    (2, 3, 1 << 19, "f32"),     # the same in fp32 (1024-logit chunks)
])
def test_maximum_sizes(B, gamma, V, dtype):
    wl = workload("chain_7b").scaled(B=B, gamma=gamma, V=V, dtype=dtype)
    lg = logits_inputs(wl, seed=gamma + V % 97)
    for offset in range(2):
        g, _, _ = _run(wl, lg, seed=41, offset=offset)
        assert g["status"] == 0


@pytest.mark.parametrize("impl", TREE_IMPLS)
@pytest.mark.parametrize("V", [64, 1001, 32000])
def test_trees(V, impl):
    # V = 1001: bf16 rows of 2002 bytes are not 16-byte vectors, so the tree
    # takes the staged kernels; the others take the cluster walk
    wl = workload("tree_64").scaled(B=6, V=V)
    lg = logits_inputs(wl, seed=3)
    for offset in range(4):
        _run(wl, lg, seed=7, offset=offset, impl=impl)


@pytest.mark.parametrize("impl", TREE_IMPLS)
def test_wide_tree_128_nodes(impl):
    # 128 nodes of a width-8 tree: child lists and draft-row selection past
    # node 64, up to 7 residual updates at one node
    wl = workload("tree_wide_128").scaled(B=6)
    lg = logits_inputs(wl, seed=14)
    assert lg["parent"].shape[1] == 128
    for offset in range(3):
        g, o, _ = _run(wl, lg, seed=13, offset=offset, impl=impl)
        assert g["status"] == 0


@pytest.mark.parametrize("impl", TREE_IMPLS)
def test_tree_walk_fp32_greedy_mix_and_shards(impl):
    # fp32 rows (the walk's float instance), every other request greedy, and
    # request shards with b_base reproducing the whole batch draw for draw
    wl = workload("tree_64").scaled(B=6, V=4096, dtype="f32")
    lg = logits_inputs(wl, seed=23)
    lg["temperature"][::2] = 0.0
    whole, _, _ = _run(wl, lg, seed=21, offset=1, impl=impl)
    assert whole["status"] == 0
    for lo, hi in [(0, 2), (2, 6)]:
        part = {k: (v[lo:hi] if isinstance(v, np.ndarray) else v) for k, v in lg.items()}
        g, _, _ = _run(wl.scaled(B=hi - lo), part, seed=21, offset=1, b_base=lo, impl=impl)
        for key in ("out_tokens", "path", "accepted_len"):
            assert np.array_equal(g[key], whole[key][lo:hi]), (key, lo)


@pytest.mark.parametrize("impl", TREE_IMPLS)
def test_single_node_and_two_level_trees(impl):
    # a tree of the root alone (the bonus draw from p of node 0, nothing
    # tested) and a three-node tree
    for nodes, depth in [(1, 0), (3, 2)]:
        wl = workload("tree_64").scaled(B=5, V=2048, gamma=depth, tree_nodes=nodes)
        lg = logits_inputs(wl, seed=24 + nodes)
        assert lg["parent"].shape[1] == nodes
        g, o, _ = _run(wl, lg, seed=22, offset=0, impl=impl)
        assert g["status"] == 0
        if nodes == 1:
            assert np.all(g["accepted_len"] == 0)


@pytest.mark.parametrize("impl", TREE_IMPLS)
def test_small_trees_many_rejections(impl):
    # wide fan-out, noisy draft: several rejections per node
    wl = workload("tree_64").scaled(B=8, V=48, gamma=2, tree_width=8,
                                    tree_nodes=40, noise=3.0)
    lg = logits_inputs(wl, seed=4)
    for offset in range(6):
        _run(wl, lg, seed=11, offset=offset, impl=impl)


@pytest.mark.parametrize("impl", IMPLS)
def test_all_accept_and_all_reject(impl):
    wl = workload("chain_7b").scaled(B=16, V=4000)
    lg = logits_inputs(wl, seed=5)
    same = dict(lg, draft=lg["target"].copy())
    g, o, _ = _run(wl, same, seed=1, offset=0, impl=impl)
    assert np.all(g["accepted_len"] == wl.gamma)
    assert np.allclose(g["probe"][:, wl.gamma, 2], 1.0)
    rej = dict(lg, target=lg["target"].copy())
    x1 = lg["tokens"][:, 1]
    rej["target"][np.arange(wl.B), 0, x1] = -np.inf
    g, o, _ = _run(wl, rej, seed=1, offset=0, impl=impl)
    assert np.all(g["accepted_len"] == 0)
    assert np.all(g["out_tokens"][:, 0] != x1)


@pytest.mark.parametrize("V,impl", [(300, sv.REJECT_AUTO), (4096, sv.REJECT_FUSED),
                                    (4096, sv.REJECT_STAGED)])
def test_failed_requests(V, impl):
    # V = 300: rows not 16-byte aligned (the staged kernels' scalar path);
    # 4096: the one-kernel path and the staged chain tail
    wl = workload("chain_7b").scaled(B=5, V=V)
    lg = logits_inputs(wl, seed=6)
    lg["target"][1, 2, 7] = np.nan
    lg["draft"][2, 0, 3] = np.inf
    lg["temperature"][3] = -1.0
    lg["tokens"][4, 2] = V
    g, o, _ = _run(wl, lg, seed=2, offset=0, impl=impl)
    assert list(g["accepted_len"][1:]) == [-1, -1, -1, -1]
    assert g["accepted_len"][0] >= 0
    assert g["status"] == (1 << 1) | (1 << 5) | (1 << 6)
    assert np.all(g["out_tokens"][1:] == -1) and np.all(g["path"][1:] == -1)


def test_gpu_output_law_chi_square():
    """10^6 independent requests: the first emitted token follows p."""
    B, gamma, V = 1_000_000, 3, 8
    rng = np.random.default_rng(12)
    z = rng.normal(0, 1.5, V)
    d = z + rng.normal(0, 1.0, V)
    q = softmax_rows(d[None], 1.0)[0]
    p = softmax_rows(z[None], 1.0)[0]
    M = gamma + 1
    lg = dict(target=np.broadcast_to(z.astype(np.float32), (B, M, V)),
              draft=np.broadcast_to(d.astype(np.float32), (B, M, V)),
              tokens=rng.choice(V, size=(B, M), p=q).astype(np.int32),
              parent=None, temperature=np.ones(B, dtype=np.float32))
    wl = workload("tiny_chain").scaled(B=B, gamma=gamma, V=V, dtype="f32")
    g = gpu_reject(wl, lg, seed=31337, offset=0, probe=False)
    counts = np.bincount(g["out_tokens"][:, 0], minlength=V)
    assert stats.chisquare(counts, p * B).pvalue > 1e-3
    alpha = np.minimum(p, q).sum()
    first = (g["accepted_len"] >= 1).mean()
    assert abs(first - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / B)
    emitted = g["accepted_len"] + 1
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(emitted.mean() - expect) < 4 * emitted.std() / np.sqrt(B)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["chain_gqa_128k", "tree_64", "stress_gqa_152k"])
def test_greedy_full_size(name, impl):
    """Temperature 0 (page 1 §4.3): exact match with each row's argmax; the
    drawn token is the argmax.  Bit-exact: no decision is near a threshold."""
    wl = workload(name)
    lg = logits_inputs(wl, seed=8)
    lg["temperature"][:] = 0.0
    # make some drafts the target's argmax so that acceptances happen
    t = lg["target"]
    for b in range(wl.B):
        for c in range(1, wl.M):
            par = c - 1 if lg["parent"] is None else lg["parent"][b, c]
            if (b + c) % 3 != 0:
                lg["tokens"][b, c] = int(np.argmax(t[b, par]))
    g, o, near = _run(wl, lg, seed=3, offset=0, impl=impl)
    assert near == 0 and g["status"] == 0
    assert np.array_equal(g["out_tokens"], o["out_tokens"])
    assert np.array_equal(g["path"], o["path"])
    assert (o["accepted_len"] > 0).any()


@pytest.mark.parametrize("impl", IMPLS)
def test_greedy_mixed_batch_and_ties(impl):
    # half the requests greedy, half sampled, in one call; a greedy row with
    # its maximum repeated (the smallest index must win)
    wl = workload("chain_7b").scaled(B=12, V=16384)
    lg = logits_inputs(wl, seed=9)
    lg["temperature"][::2] = 0.0
    t = lg["target"]
    top = bf16_round(np.array([t[0, 0].max() + 1.0], np.float32))[0]
    t[0, 0, 100] = top
    t[0, 0, 9000] = top
    lg["tokens"][0, 1] = 9000          # a tie, but not the first maximum: rejected
    g, o, _ = _run(wl, lg, seed=4, offset=2, impl=impl)
    assert g["accepted_len"][0] == 0 and g["out_tokens"][0, 0] == 100
    greedy = lg["temperature"] == 0.0
    assert np.array_equal(g["out_tokens"][greedy], o["out_tokens"][greedy])


@pytest.mark.parametrize("impl", IMPLS)
def test_request_shards_reproduce_the_whole_batch(impl):
    """Request shards on several GPUs: each shard passes the global index of
    its first request as b_base, so its uniforms, and hence its outputs,
    are those of the same requests in one whole-batch call."""
    wl = workload("chain_7b").scaled(B=10, V=16384)
    lg = logits_inputs(wl, seed=12)
    whole, _, _ = _run(wl, lg, seed=77, offset=3, impl=impl)
    for lo, hi in [(0, 4), (4, 7), (7, 10)]:
        part = {k: (v[lo:hi] if isinstance(v, np.ndarray) else v) for k, v in lg.items()}
        g, _, _ = _run(wl.scaled(B=hi - lo), part, seed=77, offset=3, b_base=lo, impl=impl)
        for key in ("out_tokens", "path", "accepted_len"):
            assert np.array_equal(g[key], whole[key][lo:hi]), (key, lo)
