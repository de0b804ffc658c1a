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
    (dict(Q=0x1008), -4), (dict(LSE=0x2002), -4), (dict(V=0x3002), -4),
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


def test_options_struct_checks(lib):
    # The options are checked before the arguments.  Every call passes a Q that is not
    # 16-byte aligned, so a call whose options are accepted stops at the alignment check
    # (-4) and none of them reaches a GPU, on any machine.
    def call(**kw):
        o = pkg.AttnOptions(ctypes.sizeof(pkg.AttnOptions), kw.get("tau", 0.0), kw.get("mode", 0), kw.get("kb", 0))
        if "size" in kw:
            o.size = kw["size"]
        return lib.attn_fwd_ex(0x10008, 0x20000, 0x30000, 0x40000, 0x50000, 1, 2, 256, 256, kw.get("d", 64), 0.125,
                               0, None, ctypes.byref(o), None)
    assert call(size=4) == -8
    assert call(tau=-1.0) == -8
    assert call(tau=21.0) == -8
    assert call(tau=float("nan")) == -8
    assert call(mode=3) == -8
    assert call(mode=-1) == -8
    assert call(kb=32) == -8                 # keys per block: 0, 64, 128 or 192
    assert call(kb=256) == -8
    assert call(kb=192, mode=2) == -8        # the 64- and 192-key builds take the hardware exponentials
    assert call(kb=64, mode=2) == -8
    # accepted options: the call gets past them to the alignment check.  A struct that
    # ends before key_block (its size was 16 bytes) is accepted and gets the default.
    assert call() == -4
    assert call(size=16) == -4
    assert call(kb=128) == -4
    assert call(kb=192, d=128) == -4
    assert call(kb=64, d=128) == -4
    assert call(tau=20.0, mode=2) == -4
    assert ctypes.sizeof(pkg.AttnOptions) == 24


def test_exp2_polynomial_bound():
    """The committed coefficients reproduce the generator's stated bound, evaluated in
    float32 the way the kernel does (Horner, one rounding per fused multiply-add); with
    the kernel's clamp, range reduction and exponent-field scaling (bit for bit, in
    wrapping 32-bit integers) the bound holds for 2^x on [-125, 29] and every argument
    below the clamp gives a finite value no larger than 2^-124."""
    import importlib.util
    import numpy as np
    path = os.path.join(ROOT, "online_softmax_flashattention_attention_gb300", "csrc")
    spec = importlib.util.spec_from_file_location("gen_exp2_poly", os.path.join(path, "gen_exp2_poly.py"))
    g = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(g)
    text = open(os.path.join(path, "exp2_poly.cuh")).read()
    c = np.array([float(re.search(rf"kExp2C{k} = ([0-9.e+-]+)f;", text).group(1)) for k in range(5)], np.float32)
    bound = float(re.search(r"kExp2PolyMaxRelError = ([0-9.e+-]+)f;", text).group(1))
    assert bound < 3e-6
    assert g.max_rel_error(c) <= bound * 1.001
    kernel = open(os.path.join(path, "attn_fwd_kernel.cuh")).read()
    lo = float(re.search(r"x\.x = fmaxf\(x\.x, (-[0-9.]+)f\);", kernel).group(1))
    assert lo == -125.0

    def kernel_exp2(x):
        x = np.maximum(x.astype(np.float32), np.float32(lo))
        t = (x + np.float32(12582912.0)).astype(np.float32)
        nj = (np.float32(12582912.0) - t).astype(np.float32)       # exact
        f = (x + nj).astype(np.float32)
        assert np.all(np.abs(f) <= 0.5)
        p = g.horner_f32(c, f)
        bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << np.uint64(23)))
        return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)

    x = np.linspace(-125.0, 29.0, 2_000_001).astype(np.float32)
    r = kernel_exp2(x).astype(np.float64)
    assert np.abs(r / np.exp2(x.astype(np.float64)) - 1.0).max() <= bound * 1.001
    below = np.concatenate([np.linspace(-1e4, -125.0, 100_001), [-np.inf]]).astype(np.float32)
    rb = kernel_exp2(below)
    assert np.all(np.isfinite(rb)) and np.all(rb >= 0) and np.all(rb <= 2.0 ** -124)
