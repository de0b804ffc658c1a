"""attn_fwd_noalloc: the entry point for callers that must not allocate device memory
(a fixed memory budget or someone else's pool, no allocation after start-up, a plugin
that must not grow its host's footprint).  Its scratch is a fixed array inside the
library instead of cudaMalloc'd memory.

Called through the C ABI with ctypes on two problems in a row (the second call reuses
the array the first one left behind); each result is compared with the fp64 oracle
under the parity tolerance of the other GPU tests, and with attn_fwd on the same inputs.
A second test runs the entry point alone in a fresh process and checks that its first
call takes no device memory.  This file is collected last on purpose.
"""
import ctypes
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, run_cuda, to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def test_noalloc_matches_oracle_and_attn_fwd_on_two_calls_in_a_row():
    lib = _lib()
    problems = [_problem(2, 3, 300, 300, 128, True, seed=41, lens=[300, 170]),
                _problem(1, 2, 256, 383, 64, False, seed=42)]
    for x in problems:
        O, LSE = _run_noalloc(lib, x)          # the allocation-free entry point
        O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], x["causal"], x["lens"])
        compare(O, LSE, O_ref, LSE_ref)
        O_fwd, LSE_fwd = run_cuda(x)            # the existing entry point, same tolerance
        compare(O, LSE, O_fwd, LSE_fwd)


def test_noalloc_rejects_bad_arguments_like_attn_fwd():
    lib = _lib()
    rc = lib.attn_fwd_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 1, 16, 16, 96, 0.1, 0, None, 1,
                              None)
    assert rc == -3


_FRESH_PROCESS = r"""
import ctypes, ctypes.util, glob, json, os, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import online_softmax_flashattention_attention_gb300 as pkg

# The CUDA runtime through ctypes rather than torch: under eager module loading torch's first
# CUDA use would load every kernel torch ships, which takes minutes; the runtime library
# registers no kernels of its own.
def cudart():
    names = [ctypes.util.find_library("cudart"), "/usr/local/cuda/lib64/libcudart.so"]
    names += sorted(glob.glob(os.path.join(sys.prefix, "lib", "python3*", "*-packages", "nvidia", "*", "lib",
                                           "libcudart.so*")))
    names += sorted(glob.glob("/usr/local/lib/python3*/dist-packages/nvidia/*/lib/libcudart.so*"))
    for n in names:
        if n:
            try:
                return ctypes.CDLL(n)
            except OSError:
                pass
    raise RuntimeError("no CUDA runtime library found")

rt = cudart()
vp, sz = ctypes.c_void_p, ctypes.c_size_t
rt.cudaMalloc.argtypes = [ctypes.POINTER(vp), sz]
rt.cudaMemcpy.argtypes = [vp, vp, sz, ctypes.c_int]
rt.cudaMemGetInfo.argtypes = [ctypes.POINTER(sz), ctypes.POINTER(sz)]
rt.cudaDeviceSynchronize.argtypes = []
for f in (rt.cudaMalloc, rt.cudaMemcpy, rt.cudaMemGetInfo, rt.cudaDeviceSynchronize):
    f.restype = ctypes.c_int

def free_bytes():
    f, t = sz(), sz()
    assert rt.cudaDeviceSynchronize() == 0 and rt.cudaMemGetInfo(ctypes.byref(f), ctypes.byref(t)) == 0
    return f.value

def device_array(host):
    p = vp()
    assert rt.cudaMalloc(ctypes.byref(p), host.nbytes) == 0
    assert rt.cudaMemcpy(p, host.ctypes.data, host.nbytes, 1) == 0   # host to device
    return p

lib = pkg.load_library()
# Load the library's device module first (its code and the fixed array): with eager module
# loading that happens at the library's first CUDA runtime call, a stream synchronisation
# here, which allocates nothing itself.
assert lib.attn_status_sync(None) == 0
f = lib.attn_fwd_noalloc
i = ctypes.c_int
f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, i, vp]
f.restype = i
rng = np.random.default_rng(3)
out = {}
for d in (128, 64):  # d = 64 with many heads takes the two-tile kernel
    H, N = (2 if d == 128 else 304), 384
    x = (rng.standard_normal((3, 1, H, N, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Q, K, V = (device_array(np.ascontiguousarray(x[t])) for t in range(3))
    O = device_array(np.zeros((1, H, N, d), np.uint16))
    L = device_array(np.zeros((1, H, N), np.float32))
    free0 = free_bytes()
    rc = f(Q, K, V, O, L, 1, H, N, N, d, d ** -0.5, 1, None, 1, None)
    free1 = free_bytes()
    o = np.zeros((1, H, N, d), np.uint16)
    assert rt.cudaMemcpy(o.ctypes.data, O, o.nbytes, 2) == 0          # device to host
    vals = (o.astype(np.uint32) << 16).view(np.float32)
    out[d] = dict(rc=rc, free_before=free0, free_after=free1, finite=bool(np.isfinite(vals).all()),
                  nonzero=bool((vals != 0).any()))
print("RESULT " + json.dumps(out))
"""


def test_noalloc_first_calls_take_no_device_memory():
    """In a fresh process, the first calls of the entry point (set-up included, at d = 128
    and d = 64) leave the device's free memory unchanged.  The library's device module (its
    code and the fixed array) is loaded before the measurement, with eager module loading
    at the library's first runtime call (a stream synchronisation); under CUDA's default
    lazy loading that load would happen at the first call of any entry point and take one
    2 MiB granule of device memory.  After it, the only change a call could make is an
    allocation of its own, and cudaMalloc hands out at least 2 MiB."""
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS, ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")]
    assert r.returncode == 0 and line, r.stdout[-2000:] + r.stderr[-2000:]
    res = json.loads(line[0][len("RESULT "):])
    for d, v in res.items():
        assert v["rc"] == 0 and v["finite"] and v["nonzero"], (d, v)
        assert v["free_before"] - v["free_after"] < (2 << 20), (d, v)
