"""The C-ABI library loads, exports every entry point include/attn.h declares, and
rejects bad arguments before touching the GPU (no device needed for these calls)."""
import ctypes
import os
import re

import pytest

import online_softmax_flashattention_attention_gb300 as pkg
from online_softmax_flashattention_attention_gb300 import build as pkgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkgbuild.build_library()
    return pkg.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    assert set(pkg.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version(lib):
    assert pkg.version() >= 100


def test_library_is_sm103a_only():
    out = open(pkg.LIB_PATH, "rb").read()
    assert b"sm_103a" in out or b"sm_103" in out


@pytest.mark.parametrize("args,status", [
    (dict(d=96), -3), (dict(d=0), -3), (dict(B=-1), -2), (dict(Nk=-5), -2), (dict(scale=0.0), -8),
    (dict(scale=-0.1), -8), (dict(scale=float("nan")), -8), (dict(scale=float("inf")), -8),
    (dict(Q=0), -1), (dict(O=0), -1), (dict(LSE=0), -1), (dict(K=0), -1), (dict(V=0), -1),
    (dict(Q=0x1008), -4), (dict(LSE=0x2004), -4), (dict(V=0x3002), -4),
])
def test_argument_errors(lib, args, status):
    a = dict(Q=0x10000, K=0x20000, V=0x30000, O=0x40000, LSE=0x50000, B=1, H=2, Nq=256, Nk=256, d=64,
             scale=0.125, causal=0, lens=None, stream=None)
    a.update(args)
    rc = pkg.attn_fwd_raw(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                          a["scale"], a["causal"], a["lens"], a["stream"])
    assert rc == status
    assert pkg.load_library().attn_last_error().decode() != ""


def test_empty_problems_are_noops(lib):
    # nothing to write: OK without any pointer or device
    for B, H, Nq in ((0, 4, 16), (2, 0, 16), (2, 4, 0)):
        assert pkg.attn_fwd_raw(None, None, None, None, None, B, H, Nq, 16, 64, 0.125, 0, None, None) == 0
    # Nk == 0 still needs the outputs (every row is written as fully masked)
    assert pkg.attn_fwd_raw(None, None, None, None, None, 1, 1, 4, 0, 64, 0.125, 0, None, None) == -1
