"""Stream order under programmatic dependent launch.

Every kernel is launched so that it may start on the SMs the previous kernel in its
stream has left and wait, before its first global-memory access, for that kernel to
finish.  These tests chain calls in one stream with no synchronisation between them,
each call reading what the one before wrote (read after write) or overwriting what the
one before reads (write after read), and compare the bytes with the same chain run
with a device synchronisation after every call.  The outputs are deterministic, so any
difference means a kernel touched memory out of stream order.  The smallest shape runs
4 CTAs on a GPU of 152 SMs: the next launch's CTAs start at once on idle SMs, where an
early read would show.  Every chain's first call is also checked against the oracle.
"""
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, to_device

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, N, d, causal
    (1, 2, 256, 64, False),     # 4 CTAs: the dependent launch lands on idle SMs at once
    (2, 16, 1024, 128, True),   # one-tile kernel, rank-major order
    (2, 80, 512, 64, True),     # two-tile kernel
]


def inputs(B, H, N, d, causal, seed):
    w = dict(name="custom", B=B, H=H, Nq=N, Nk=N, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None, plant=None, scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def chain(Q, K, V, causal, scale, sync):
    """Five calls back to back (outputs filled with NaN before the first):
    O1 = f(Q, K, V); O2 = f(Q, K, O1); O3 = f(O2, O1, V); O4 = f(O3, K, O1); and last
    O1 = f(Q, K, O3), which overwrites O1 while the call before it reads O1.  With
    `sync`, a device synchronisation follows every call and the first call's O and LSE
    are kept."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    B, H, N, _ = Q.shape
    O1, O2, O3, O4 = (torch.full_like(Q, float("nan")) for _ in range(4))
    LSE1 = torch.full((B, H, N), float("nan"), device=Q.device)
    torch.cuda.synchronize()
    first = None
    calls = [(Q, K, V, O1, LSE1), (Q, K, O1, O2, None), (O2, O1, V, O3, None), (O3, K, O1, O4, None),
             (Q, K, O3, O1, None)]
    for i, (q, k, v, o, lse) in enumerate(calls):
        pkg.attn_fwd(q, k, v, o, lse, scale=scale, causal=causal)
        if sync:
            torch.cuda.synchronize()
            if i == 0:
                first = (O1.float().cpu().numpy().astype(np.float64), LSE1.cpu().numpy().astype(np.float64))
    pkg.status_sync()
    return [t.float().cpu().numpy() for t in (O2, O3, O4, O1)], first


@pytest.mark.parametrize("B,H,N,d,causal", SHAPES)
def test_chained_calls_keep_stream_order(B, H, N, d, causal):
    x = inputs(B, H, N, d, causal, seed=2300 + d + N)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    ref, first = chain(Q, K, V, causal, x["scale"], sync=True)
    O_ref, L_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, None)
    compare(first[0], first[1], O_ref, L_ref)
    assert not np.array_equal(ref[3], first[0].astype(np.float32)), "the last call must change O1"
    for rep in range(5):
        got, _ = chain(Q, K, V, causal, x["scale"], sync=False)
        for i, (a, b) in enumerate(zip(got, ref)):
            assert not np.isnan(a).any(), (rep, i)
            assert np.array_equal(a, b), (rep, i)


def test_splitkv_chain_keeps_stream_order():
    """The split-KV route launches two kernels per call (states, then their merge); a
    second call reads the first call's O as its V."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    x = inputs(1, 8, 640, 128, True, seed=2400)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])

    def run(sync):
        O1, O2 = torch.full_like(Q, float("nan")), torch.full_like(Q, float("nan"))
        torch.cuda.synchronize()
        pkg.attn_fwd_splitkv(Q, K, V, O1, num_splits=3, scale=x["scale"], causal=True)
        if sync:
            torch.cuda.synchronize()
        pkg.attn_fwd_splitkv(Q, K, O1, O2, num_splits=3, scale=x["scale"], causal=True)
        pkg.status_sync()
        return O1.float().cpu().numpy(), O2.float().cpu().numpy()

    ref1, ref2 = run(sync=True)
    for _ in range(5):
        a1, a2 = run(sync=False)
        assert not np.isnan(a2).any()
        assert np.array_equal(a1, ref1) and np.array_equal(a2, ref2)
