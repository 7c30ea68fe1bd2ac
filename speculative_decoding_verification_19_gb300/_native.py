"""ctypes binding of libspecverify.so (argument marshalling only).

Every function here takes torch tensors that already live on the GPU,
passes their device pointers, sizes and the current CUDA stream to the C ABI
declared in include/spec_verify.h, and raises SpecError on a non-zero status.
No step of the verify path runs in Python.  If the shared library is missing
the import fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SPEC_BF16, SPEC_F32 = 0, 1
STATUS_NAMES = {
    0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_CAPACITY",
    3: "SPEC_ERR_UNSUPPORTED", 4: "SPEC_ERR_CUDA", 5: "SPEC_ERR_NONFINITE",
    6: "SPEC_ERR_DEVICE_BOUNDS", 7: "SPEC_ERR_TIMEOUT",
}
ATTN_AUTO, ATTN_CUDA_CORES, ATTN_TENSOR_CORES = 0, 1, 2
REJECT_AUTO, REJECT_STAGED, REJECT_FUSED = 0, 1, 2

# every symbol the header declares
EXPORTS = (
    "spec_workspace_size", "spec_workspace_init", "spec_get_device_status",
    "spec_verify_attn", "spec_reject_sample", "spec_reject_sample_filtered", "kv_commit",
    "spec_philox_block", "spec_lm_head", "spec_reject_sample_lm_head",
    "spec_status_string", "spec_last_launch_count", "spec_reject_sample_noalloc",
    "spec_ctrl_default_config", "spec_ctrl_init", "spec_ctrl_update", "spec_ctrl_metrics",
    "spec_step_stats",
)


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


class SpecDims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("M", ctypes.c_int32), ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("block", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("V", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("logits_dtype", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
        ("attn_impl", ctypes.c_int32), ("reject_impl", ctypes.c_int32),
        ("wait_limit_kcycles", ctypes.c_int32),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_uint64
    pd = ctypes.POINTER(SpecDims)
    L.spec_workspace_size.argtypes = [pd]
    L.spec_workspace_size.restype = sz
    L.spec_workspace_init.argtypes = [vp, sz, vp]
    L.spec_workspace_init.restype = i32
    L.spec_get_device_status.argtypes = [vp, vp, ctypes.POINTER(i32), i32]
    L.spec_get_device_status.restype = i32
    L.spec_verify_attn.argtypes = [vp] * 10 + [pd, vp, sz, vp]
    L.spec_verify_attn.restype = i32
    L.spec_reject_sample.argtypes = [vp, vp, vp, vp, vp, u64, u64, u64, vp, vp, vp,
                                     vp, pd, vp, sz, vp]
    L.spec_reject_sample.restype = i32
    L.spec_reject_sample_filtered.argtypes = [vp, vp, vp, vp, vp, vp, vp, u64, u64, u64, vp,
                                              vp, vp, vp, pd, vp, sz, vp]
    L.spec_reject_sample_filtered.restype = i32
    L.spec_lm_head.argtypes = [vp, vp, i32, i32, i32, vp, vp, sz, vp]
    L.spec_lm_head.restype = i32
    L.spec_reject_sample_lm_head.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, u64,
                                             u64, u64, vp, vp, vp, vp, pd, vp, sz, vp]
    L.spec_reject_sample_lm_head.restype = i32
    L.spec_reject_sample_noalloc.argtypes = [vp, vp, vp, vp, vp, u64, u64, u64, vp, vp,
                                             vp, vp, pd, vp]
    L.spec_reject_sample_noalloc.restype = i32
    L.kv_commit.argtypes = [vp] * 7 + [pd, vp, sz, vp]
    L.kv_commit.restype = i32
    L.spec_philox_block.argtypes = [ctypes.POINTER(u64)] * 3
    L.spec_philox_block.restype = None
    L.spec_status_string.argtypes = [i32]
    L.spec_status_string.restype = ctypes.c_char_p
    L.spec_last_launch_count.argtypes = []
    L.spec_last_launch_count.restype = i32
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise SpecError(fn, code)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return SPEC_BF16
    if dt == torch.float32:
        return SPEC_F32
    raise ValueError(f"unsupported dtype {dt}")


def make_dims(B, M, Hq=1, Hkv=1, D=128, max_blocks=1, num_blocks=1, V=1,
              kv_dtype=torch.bfloat16, logits_dtype=torch.bfloat16,
              softmax_scale=0.0, block=16, attn_impl=0, reject_impl=0,
              wait_limit_kcycles=0) -> SpecDims:
    return SpecDims(B, M, Hq, Hkv, D, block, max_blocks, num_blocks, V,
                    dtype_code(kv_dtype), dtype_code(logits_dtype),
                    float(softmax_scale), int(attn_impl), int(reject_impl),
                    int(wait_limit_kcycles))


def workspace_size(dims: SpecDims) -> int:
    return int(lib().spec_workspace_size(ctypes.byref(dims)))


def workspace(dims: SpecDims, device="cuda", stream=None) -> torch.Tensor:
    """A zero-initialised device workspace for calls with these dims."""
    n = workspace_size(dims)
    if n == 0:
        raise SpecError("spec_workspace_size", 1)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check("spec_workspace_init",
           lib().spec_workspace_init(_ptr(ws), n, _stream(stream)))
    return ws


def device_status(ws: torch.Tensor, clear: bool = True, stream=None) -> int:
    """Bitmask of spec_status codes raised on the device (syncs the stream)."""
    out = ctypes.c_int32(0)
    _check("spec_get_device_status",
           lib().spec_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(out),
                                        1 if clear else 0))
    return int(out.value)


def spec_verify_attn(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens,
                     parent, out, lse, dims: SpecDims, ws, stream=None) -> int:
    code = lib().spec_verify_attn(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), _ptr(ctx_lens), _ptr(parent), _ptr(out), _ptr(lse),
        ctypes.byref(dims), _ptr(ws), ws.numel(), _stream(stream))
    _check("spec_verify_attn", code)
    return lib().spec_last_launch_count()


def spec_reject_sample(target_logits, draft_logits, tokens, parent, temperature,
                       seed, offset, out_tokens, path, accepted_len, probe,
                       dims: SpecDims, ws, b_base=0, stream=None, top_k=None,
                       top_p=None) -> int:
    """spec_reject_sample; with top_k and / or top_p ([B] int32 / float32
    device tensors) spec_reject_sample_filtered."""
    if top_k is None and top_p is None:
        code = lib().spec_reject_sample(
            _ptr(target_logits), _ptr(draft_logits), _ptr(tokens), _ptr(parent),
            _ptr(temperature), int(seed) % (1 << 64), int(offset) % (1 << 64),
            int(b_base) % (1 << 64), _ptr(out_tokens), _ptr(path), _ptr(accepted_len),
            _ptr(probe), ctypes.byref(dims), _ptr(ws), ws.numel(), _stream(stream))
        _check("spec_reject_sample", code)
    else:
        code = lib().spec_reject_sample_filtered(
            _ptr(target_logits), _ptr(draft_logits), _ptr(tokens), _ptr(parent),
            _ptr(temperature), _ptr(top_k), _ptr(top_p), int(seed) % (1 << 64),
            int(offset) % (1 << 64), int(b_base) % (1 << 64), _ptr(out_tokens), _ptr(path),
            _ptr(accepted_len), _ptr(probe), ctypes.byref(dims), _ptr(ws), ws.numel(),
            _stream(stream))
        _check("spec_reject_sample_filtered", code)
    return lib().spec_last_launch_count()


def spec_lm_head(hidden, weight, logits, ws, stream=None) -> int:
    """logits [rows, V] = hidden [rows, H] @ weight [V, H]^T (bf16)."""
    rows, H = hidden.shape
    V = weight.shape[0]
    code = lib().spec_lm_head(_ptr(hidden), _ptr(weight), rows, H, V, _ptr(logits), _ptr(ws),
                              ws.numel(), _stream(stream))
    _check("spec_lm_head", code)
    return lib().spec_last_launch_count()


def spec_reject_sample_lm_head(hidden_target, weight_target, hidden_draft, weight_draft,
                               target_logits, draft_logits, tokens, parent, temperature, seed,
                               offset, out_tokens, path, accepted_len, probe, dims: SpecDims, ws,
                               b_base=0, stream=None) -> int:
    """The target and draft LM heads with the verify decisions (the
    statistics formed in the LM heads' epilogue)."""
    code = lib().spec_reject_sample_lm_head(
        _ptr(hidden_target), _ptr(weight_target), hidden_target.shape[-1], _ptr(hidden_draft),
        _ptr(weight_draft), hidden_draft.shape[-1], _ptr(target_logits), _ptr(draft_logits),
        _ptr(tokens), _ptr(parent), _ptr(temperature), int(seed) % (1 << 64),
        int(offset) % (1 << 64), int(b_base) % (1 << 64), _ptr(out_tokens), _ptr(path),
        _ptr(accepted_len), _ptr(probe), ctypes.byref(dims), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("spec_reject_sample_lm_head", code)
    return lib().spec_last_launch_count()


def spec_reject_sample_noalloc(target_logits, draft_logits, tokens, parent,
                               temperature, seed, offset, out_tokens, path,
                               accepted_len, probe, dims: SpecDims, b_base=0,
                               stream=None) -> None:
    """spec_reject_sample without a workspace, for callers that cannot
    allocate device memory; its scratch is a fixed 1 MiB array inside the
    library shared by every call, so overlapping calls race."""
    code = lib().spec_reject_sample_noalloc(
        _ptr(target_logits), _ptr(draft_logits), _ptr(tokens), _ptr(parent),
        _ptr(temperature), int(seed) % (1 << 64), int(offset) % (1 << 64),
        int(b_base) % (1 << 64), _ptr(out_tokens), _ptr(path), _ptr(accepted_len),
        _ptr(probe), ctypes.byref(dims), _stream(stream))
    _check("spec_reject_sample_noalloc", code)


def kv_commit(k_cache, v_cache, block_table, ctx_lens, new_ctx_lens, path,
              accepted_len, dims: SpecDims, ws, stream=None) -> int:
    code = lib().kv_commit(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens),
        _ptr(new_ctx_lens), _ptr(path), _ptr(accepted_len), ctypes.byref(dims),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("kv_commit", code)
    return lib().spec_last_launch_count()


def philox_block(key, counter):
    """Host-side Philox4x64-10 block of the library (for known-answer tests)."""
    K = (ctypes.c_uint64 * 2)(*[int(k) % (1 << 64) for k in key])
    C = (ctypes.c_uint64 * 4)(*[int(c) % (1 << 64) for c in counter])
    O = (ctypes.c_uint64 * 4)()
    lib().spec_philox_block(K, C, O)
    return [int(x) for x in O]
