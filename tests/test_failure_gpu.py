"""Failure detection on the GPU without a fault: a test hook makes the producer withhold
one K block, so the waits on it run out after a short limit.  The kernel must end on its
own, report ATTN_ERR_TIMEOUT through the status word, and leave the context usable: the
next call returns correct results."""
import ctypes
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, run_cuda, to_device

pytestmark = pytest.mark.gpu


def _problem(seed):
    w = dict(name="fail", B=1, H=2, Nq=512, Nk=512, d=128, causal=False, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None, plant=None, scale=1.0 / math.sqrt(128))
    return gen.make_inputs(w)


def test_withheld_block_times_out_and_context_survives(monkeypatch):
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    x = _problem(51)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((1, 2, 512), dtype=torch.float32, device="cuda")
    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "100")
    monkeypatch.setenv("ATTN_ENABLE_TEST_HOOKS", "1")
    monkeypatch.setenv("ATTN_TEST_WITHHOLD_K_BLOCK", "1")
    pkg.attn_fwd(Q, K, V, O, LSE, scale=x["scale"])          # the launch itself succeeds
    with pytest.raises(pkg.AttnError) as err:
        pkg.status_sync()
    assert err.value.status == -7                            # ATTN_ERR_TIMEOUT
    pkg.status_sync()                                        # the word was cleared
    monkeypatch.delenv("ATTN_TEST_WITHHOLD_K_BLOCK")
    monkeypatch.delenv("ATTN_WAIT_LIMIT_MS")
    O2, LSE2 = run_cuda(x)                                   # same context, normal call
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    compare(O2, LSE2, O_ref, LSE_ref)


def test_withheld_block_reported_by_the_synchronous_noalloc_call(monkeypatch):
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    lib = pkg.load_library()
    f = lib.attn_fwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, i, vp]
    f.restype = i
    x = _problem(52)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((1, 2, 512), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "100")
    monkeypatch.setenv("ATTN_ENABLE_TEST_HOOKS", "1")
    monkeypatch.setenv("ATTN_TEST_WITHHOLD_K_BLOCK", "2")
    rc = f(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), 1, 2, 512, 512, 128,
           x["scale"], 0, None, 1, stream)
    assert rc == -7
    monkeypatch.delenv("ATTN_TEST_WITHHOLD_K_BLOCK")
    rc = f(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), 1, 2, 512, 512, 128,
           x["scale"], 0, None, 1, stream)
    assert rc == 0
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)


def test_withhold_hook_ignored_without_the_enable_switch(monkeypatch):
    """A stray ATTN_TEST_WITHHOLD_K_BLOCK in the environment must not drop keys: the hook
    acts only together with ATTN_ENABLE_TEST_HOOKS=1."""
    import online_softmax_flashattention_attention_gb300 as pkg
    x = _problem(53)
    monkeypatch.delenv("ATTN_ENABLE_TEST_HOOKS", raising=False)
    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "100")
    monkeypatch.setenv("ATTN_TEST_WITHHOLD_K_BLOCK", "1")
    O, LSE = run_cuda(x)                                     # run_cuda checks attn_status_sync
    pkg.status_sync()
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    compare(O, LSE, O_ref, LSE_ref)


def test_async_noalloc_timeout_reported_by_status_sync(monkeypatch):
    """check_status = 0: the no-alloc call returns at once; a wait that ran out is
    reported later by attn_status_sync, which also clears the fixed status word."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    lib = pkg.load_library()
    f = lib.attn_fwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, i, vp]
    f.restype = i
    x = _problem(54)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((1, 2, 512), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "100")
    monkeypatch.setenv("ATTN_ENABLE_TEST_HOOKS", "1")
    monkeypatch.setenv("ATTN_TEST_WITHHOLD_K_BLOCK", "1")
    rc = f(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), 1, 2, 512, 512, 128,
           x["scale"], 0, None, 0, stream)
    assert rc == 0                                           # asynchronous: nothing to report yet
    with pytest.raises(pkg.AttnError) as err:
        pkg.status_sync()
    assert err.value.status == -7
    pkg.status_sync()                                        # cleared by the read
    monkeypatch.delenv("ATTN_TEST_WITHHOLD_K_BLOCK")
    rc = f(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), 1, 2, 512, 512, 128,
           x["scale"], 0, None, 1, stream)
    assert rc == 0
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)
