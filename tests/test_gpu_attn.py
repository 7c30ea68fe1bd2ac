"""GPU parity of spec_verify_attn (KV append + masked verify attention).

Outputs within 2e-2 absolute + 1e-2 relative of the fp64 oracle, log-sum-exp
within 1e-3; the appended cache bit-exact (new rows at ctx..ctx+M-1, rest of
the last block zero, everything else untouched).  Every case runs on each
kernel that supports its shape (CUDA cores; tcgen05 tensor cores).  Covers
chains and trees, GQA groups 1/4/8, fp32 and bf16, contexts that are empty,
ragged or cross a block boundary, long contexts, rows per KV head from 1 to
128, more CTAs than tiles, and the device-side failure paths.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import speculative_decoding_verification_19_gb300 as sv  # noqa: E402
from harness import (assert_attn_close, dims_for, gpu_attn,  # noqa: E402
                     impls_for, oracle_attn)
from synth import kv_inputs_host, logits_inputs, workload  # noqa: E402


def _check(wl, kv, parent=None, impls=None):
    o_out, o_lse, o_kc, o_vc = oracle_attn(wl, kv, parent)
    impls = impls_for(wl) if impls is None else impls
    assert impls
    for impl in impls:
        g = gpu_attn(wl, kv, parent, impl=impl)
        assert g["status"] == 0, impl
        assert_attn_close(g["out"], o_out, g["lse"], o_lse)
        assert np.array_equal(g["k_cache"], o_kc.astype(np.float32)), impl
        assert np.array_equal(g["v_cache"], o_vc.astype(np.float32)), impl


def test_tiny_chain_full():
    wl = workload("tiny_chain")
    _check(wl, kv_inputs_host(wl, seed=0))


@pytest.mark.parametrize("name,B", [("chain_7b", 2), ("chain_gqa_128k", 3),
                                    ("stress_gqa_152k", 2)])
def test_chain_workloads(name, B):
    wl = workload(name)
    _check(wl, kv_inputs_host(wl, seed=1, B=B))


def test_tree_workload():
    wl = workload("tree_64")
    kv = kv_inputs_host(wl, seed=2, B=2)
    parent = logits_inputs(wl.scaled(V=16), seed=2, B=2)["parent"]
    _check(wl, kv, parent)


@pytest.mark.parametrize("ctx", [[0, 1, 15, 16, 17, 31], [5, 250, 1000, 4095, 33, 64]])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_contexts(ctx, dtype):
    wl = workload("chain_gqa_128k").scaled(dtype=dtype, gamma=3)
    _check(wl, kv_inputs_host(wl, seed=3, B=len(ctx), ctx=np.array(ctx)))


@pytest.mark.parametrize("Hq,Hkv,gamma", [(8, 8, 0), (8, 2, 7), (16, 2, 7), (4, 1, 15),
                                          (16, 1, 7), (32, 2, 7)])
def test_group_shapes(Hq, Hkv, gamma):
    wl = workload("chain_7b").scaled(Hq=Hq, Hkv=Hkv, gamma=gamma)
    _check(wl, kv_inputs_host(wl, seed=4, B=2, ctx=np.array([77, 300])))


def test_more_ctas_than_tiles():
    # a handful of 64-key tiles spread over one CTA per SM
    wl = workload("chain_gqa_128k").scaled(Hq=8, Hkv=2)
    _check(wl, kv_inputs_host(wl, seed=11, B=3, ctx=np.array([0, 60, 130])))


def test_many_requests():
    # more requests than the tensor-core plan keeps in shared memory (1024),
    # with mixed short contexts so that CTA ranges cross many requests
    wl = workload("chain_gqa_128k").scaled(Hq=8, Hkv=2, gamma=3)
    rng = np.random.default_rng(13)
    ctx = rng.integers(0, 200, size=1100)
    _check(wl, kv_inputs_host(wl, seed=13, B=1100, ctx=ctx), impls=[sv.ATTN_TENSOR_CORES])


def test_pairs_over_many_ctas():
    # one long request: each (request, KV head) pair spans about twenty CTAs,
    # so the CTA holding a pair's first tile merges many partials
    wl = workload("chain_gqa_128k").scaled(gamma=3)
    _check(wl, kv_inputs_host(wl, seed=14, B=1, ctx=np.array([40000])),
           impls=[sv.ATTN_TENSOR_CORES])


def test_tree_rows_up_to_128():
    wl = workload("tree_64").scaled(Hq=4, Hkv=2, tree_nodes=64, tree_width=4)
    kv = kv_inputs_host(wl, seed=12, B=2, ctx=np.array([200, 1999]))
    parent = logits_inputs(wl.scaled(V=16), seed=12, B=2)["parent"]
    _check(wl, kv, parent, impls=[sv.ATTN_TENSOR_CORES])


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f32")])
def test_wide_tree_128_nodes(D, dtype):
    # 128 nodes: ancestor masks past 64 bits, on each kernel that takes the
    # shape (128 rows per KV head)
    wl = workload("tree_wide_128").scaled(D=D, dtype=dtype, Hq=2, Hkv=2)
    kv = kv_inputs_host(wl, seed=15, B=2, ctx=np.array([0, 1500]))
    parent = logits_inputs(wl.scaled(V=16), seed=15, B=2)["parent"]
    assert parent.shape == (2, 128)  # nodes 64..127: mask bits past the first word
    _check(wl, kv, parent)


def test_more_rows_than_a_kernel_takes():
    # 128 nodes x 2 query heads per KV head = 256 rows: refused before launch
    wl = workload("tree_wide_128").scaled(Hq=4, Hkv=2)
    kv = kv_inputs_host(wl, seed=16, B=1, ctx=np.array([100]))
    parent = logits_inputs(wl.scaled(V=16), seed=16, B=1)["parent"]
    with pytest.raises(sv.SpecError) as e:
        gpu_attn(wl, kv, parent)
    assert e.value.code == 3  # SPEC_ERR_UNSUPPORTED


def test_small_head_dim_tree():
    wl = workload("tree_64").scaled(D=64, Hq=4, Hkv=2, tree_nodes=21, gamma=3)
    kv = kv_inputs_host(wl, seed=5, B=3, ctx=np.array([0, 40, 129]))
    parent = logits_inputs(wl.scaled(V=16), seed=5, B=3)["parent"]
    _check(wl, kv, parent)


@pytest.mark.parametrize("impl", [sv.ATTN_CUDA_CORES, sv.ATTN_TENSOR_CORES])
def test_capacity_and_bad_block(impl):
    wl = workload("chain_7b").scaled(Hq=4, Hkv=4, gamma=3)
    kv = kv_inputs_host(wl, seed=6, B=3, ctx=np.array([20, 40, 60]))
    kv["ctx_lens"] = kv["ctx_lens"].copy()
    kv["block_table"] = kv["block_table"].copy()
    # request 1 claims more context than its table can hold
    kv["ctx_lens"][1] = kv["max_blocks"] * 16 - 2
    # request 2 points one of its blocks outside the cache
    kv["block_table"][2, 1] = kv["num_blocks"] + 5
    g = gpu_attn(wl, kv, impl=impl)
    assert g["status"] == (1 << 2) | (1 << 6)
    assert np.all(g["out"][1:] == 0) and np.all(np.isneginf(g["lse"][1:]))
    # request 0 is unaffected; failed requests leave the cache untouched
    good = dict(kv, block_table=kv["block_table"][:1], ctx_lens=kv["ctx_lens"][:1],
                q=kv["q"][:1], k_new=kv["k_new"][:1], v_new=kv["v_new"][:1])
    o_out, o_lse, o_kc, o_vc = oracle_attn(wl, good)
    assert_attn_close(g["out"][:1], o_out, g["lse"][:1], o_lse)
    assert np.array_equal(g["k_cache"], o_kc.astype(np.float32))


def test_host_validation():
    wl = workload("chain_7b")
    dims = dims_for(wl, 1, 4, 4)
    bad = sv.make_dims(B=1, M=6, Hq=32, Hkv=5, D=128, max_blocks=4, num_blocks=4)
    assert sv.workspace_size(bad) > 0  # size is shape-only; the call rejects it
    ws = sv.workspace(dims)
    t = torch.zeros(1, 6, 32, 128, dtype=torch.bfloat16, device="cuda")
    kvn = torch.zeros(1, 6, 32, 128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(4, 32, 16, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    ctx = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_attn(t, kvn, kvn, cache, cache, bt, ctx, None, t, None, bad, ws)
    assert e.value.code == 1
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_attn(t, kvn, kvn, cache, cache, bt, ctx, None, t, None, dims,
                            ws[: ws.numel() // 2])
    assert e.value.code == 1
    # a shape no kernel supports: 200 rows per KV head
    big = sv.make_dims(B=1, M=25, Hq=8, Hkv=1, D=128, max_blocks=4, num_blocks=4)
    ws2 = sv.workspace(big)
    q2 = torch.zeros(1, 25, 8, 128, dtype=torch.bfloat16, device="cuda")
    kv2 = torch.zeros(1, 25, 1, 128, dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros(4, 1, 16, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_attn(q2, kv2, kv2, c2, c2, bt, ctx, None, q2, None, big, ws2)
    assert e.value.code == 3
    assert sv.device_status(ws) == 0
