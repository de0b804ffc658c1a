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


# ---- split-KV entry points: argument checks and workspace sizes (no device needed)

def _states_call(lib, **kw):
    a = dict(Q=0x10000, K=0x20000, V=0x30000, o=0x40000, m=0x50000, l=0x60000, B=1, H=2, Nq=256, Nk=512, d=128,
             scale=0.125, causal=0, lens=None, S=2, stream=None)
    a.update(kw)
    return lib.attn_fwd_states(a["Q"], a["K"], a["V"], a["o"], a["m"], a["l"], a["B"], a["H"], a["Nq"], a["Nk"],
                               a["d"], a["scale"], a["causal"], a["lens"], a["S"], a["stream"])


@pytest.mark.parametrize("args,status", [
    (dict(S=0), -8), (dict(S=257), -8), (dict(S=-3), -8), (dict(d=96), -3), (dict(l=0), -1), (dict(o=0), -1),
    (dict(l=0x60004), -4), (dict(o=0x40008), -4), (dict(scale=0.0), -8),
])
def test_states_argument_errors(lib, args, status):
    assert _states_call(lib, **args) == status


def _merge_call(lib, **kw):
    a = dict(o=0x10000, m=0x20000, l=0x30000, S=3, rows=100, d=128, O=0x40000, LSE=0x50000, stream=None)
    a.update(kw)
    return lib.attn_merge_states(a["o"], a["m"], a["l"], a["S"], a["rows"], a["d"], a["O"], a["LSE"], a["stream"])


@pytest.mark.parametrize("args,status", [
    (dict(d=32), -3), (dict(S=0), -8), (dict(rows=-1), -2), (dict(o=0), -1), (dict(LSE=0), -1),
    (dict(o=0x10004), -4), (dict(O=0x40002), -4), (dict(m=0x20001), -4),
])
def test_merge_argument_errors(lib, args, status):
    assert _merge_call(lib, **args) == status


def test_merge_of_no_rows_is_a_noop(lib):
    assert _merge_call(lib, rows=0, o=None, m=None, l=None, O=None, LSE=None) == 0


def test_splitkv_workspace_bytes(lib):
    f = lib.attn_splitkv_workspace_bytes
    rows = 2 * 4 * 300 * 3
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert f(2, 4, 300, 128, 3) == up(rows * 128 * 4) + 2 * up(rows * 4)
    assert f(2, 4, 300, 64, 3) == up(rows * 64 * 4) + 2 * up(rows * 4)
    assert f(2, 4, 300, 96, 3) == 0 and f(2, 4, 300, 128, 0) == 0 and f(-1, 4, 300, 128, 2) == 0


def test_splitkv_workspace_checks(lib):
    def call(ws, ws_bytes, S=4):
        return lib.attn_fwd_splitkv(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 2, 128, 4096, 128, 0.125, 0,
                                    None, S, ws, ws_bytes, None)
    need = lib.attn_splitkv_workspace_bytes(1, 2, 128, 128, 4)
    assert call(None, need) == -1
    assert call(0x70008, need) == -4
    assert call(0x70000, need - 1) == -8
    assert call(0x70000, need, S=300) == -8
