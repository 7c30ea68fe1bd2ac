"""The C ABI library builds, loads without a GPU, and exports every function
declared in include/spec_verify.h; its host-side Philox reproduces the
published known-answer vectors.  No GPU compute is called here."""
import os
import re

import pytest

import speculative_decoding_verification_19_gb300 as sv
from speculative_decoding_verification_19_gb300 import build as sv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sv_build.build()
    return sv.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "defined"):
                names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert {"spec_verify_attn", "spec_reject_sample", "kv_commit"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(sv.EXPORTS) == declared


def test_philox_known_answers(lib, golden_dir):
    with open(os.path.join(golden_dir, "philox4x64_10_kat.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for r in rows:
        w = [int(x, 16) for x in r]
        assert sv.philox_block(w[4:6], w[0:4]) == w[6:10]


def test_library_philox_matches_oracle_uniforms(lib):
    from oracle import philox_block
    for n, b, off in [(1, 0, 0), (5, 17, 3), (64, 127, 1 << 40)]:
        got = sv.philox_block([123456789, 0], [n, b, off, 0])
        assert got == [int(x) for x in philox_block(123456789, (n, b, off, 0))]


def test_workspace_size_and_status_strings(lib):
    d = sv.make_dims(B=128, M=5, Hq=64, Hkv=8, D=128, max_blocks=2049,
                     num_blocks=150000, V=152064)
    n = sv.workspace_size(d)
    assert n > 0 and n % 256 == 0
    bad = sv.make_dims(B=0, M=5)
    assert sv.workspace_size(bad) == 0
    assert lib.spec_status_string(2) == b"SPEC_ERR_CAPACITY"
