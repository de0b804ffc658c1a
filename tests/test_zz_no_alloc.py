"""attn_fwd_noalloc: the entry point for callers that must not allocate device memory
(a fixed memory budget or someone else's pool, no allocation after start-up, a plugin
that must not grow its host's footprint).  Its scratch is a fixed array inside the
library instead of cudaMalloc'd memory.

Called through the C ABI with ctypes and compared with attn_fwd, under the parity
tolerance of the other GPU tests, on two calls in a row (the second call reuses the
array the first one left behind).  This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest

import gen
from gpu_helpers import compare, run_cuda, to_device

pytestmark = pytest.mark.gpu


def _lib():
    import online_softmax_flashattention_attention_gb300 as pkg
    from online_softmax_flashattention_attention_gb300 import build as pkgbuild
    pkgbuild.build_library()
    lib = pkg.load_library()
    f = lib.attn_fwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, i, vp]
    f.restype = i
    return lib


def _problem(B, H, Nq, Nk, d, causal, seed, lens=None):
    w = dict(name="noalloc", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None if lens is None else ("given", lens), plant=None,
             scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def _run_noalloc(lib, x):
    import torch
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    B, H, Nq, d = Q.shape
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=Q.device)
    lens = None if x["lens"] is None else torch.as_tensor(np.asarray(x["lens"], np.int32)).cuda()
    stream = torch.cuda.current_stream()
    rc = lib.attn_fwd_noalloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H, Nq,
                              K.shape[2], d, x["scale"], int(x["causal"]),
                              None if lens is None else lens.data_ptr(), 1, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, lib.attn_last_error().decode()
    torch.cuda.synchronize()
    return O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64)


def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row():
    lib = _lib()
    problems = [_problem(2, 3, 300, 300, 128, True, seed=41, lens=[300, 170]),
                _problem(1, 2, 256, 383, 64, False, seed=42)]
    for x in problems:
        O_ref, LSE_ref = run_cuda(x)          # the existing entry point
        O, LSE = _run_noalloc(lib, x)         # the allocation-free one
        compare(O, LSE, O_ref, LSE_ref)


def test_noalloc_rejects_bad_arguments_like_attn_fwd():
    lib = _lib()
    rc = lib.attn_fwd_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 1, 16, 16, 96, 0.1, 0, None, 1,
                              None)
    assert rc == -3
