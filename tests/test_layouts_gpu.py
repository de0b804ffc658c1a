"""Other layouts through the C ABI against the fp64 oracle: strided tensors (the
[B, N, H, d] layout and padded rows) and packed sequences of different lengths.

The oracle is the same three-pass attention per (batch, head); the tests only move the
generator's bytes into the layout under test and back.  Each layout is also compared
bit for bit with the contiguous entry point on the same values: only the addressing
differs, so the arithmetic must be identical.
"""
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, to_device

pytestmark = pytest.mark.gpu


def _pkg():
    import online_softmax_flashattention_attention_gb300 as pkg
    return pkg


def custom(B, H, Nq, Nk, d, causal=False, seed=7, lens=None):
    w = dict(name="custom", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None if lens is None else ("given", lens), plant=None,
             scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def bshd_view(codes):
    """The [B, H, N, d] codes stored as a [B, N, H, d] tensor, viewed back as [B, H, N, d]."""
    t = to_device(codes)                        # [B, H, N, d] contiguous
    return t.transpose(1, 2).contiguous().transpose(1, 2)


STRIDED = [
    (2, 3, 300, 300, 128, True, None),
    (2, 2, 129, 257, 64, False, None),
    (3, 2, 260, 700, 128, False, [0, 1, 700]),
    (1, 4, 200, 383, 128, True, None),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,lens", STRIDED)
def test_bshd_matches_oracle_and_contiguous(B, H, Nq, Nk, d, causal, lens):
    import torch
    pkg = _pkg()
    x = custom(B, H, Nq, Nk, d, causal, seed=Nq * 3 + Nk + d, lens=lens)
    Q, K, V = bshd_view(x["Q"]), bshd_view(x["K"]), bshd_view(x["V"])
    assert Q.stride() == (Nq * H * d, d, H * d, 1)
    lt = None if lens is None else torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    O, LSE = pkg.attn_fwd_strided(Q, K, V, scale=x["scale"], causal=causal, key_padding_lens=lt)
    pkg.status_sync()
    Of = O.float().cpu().numpy().astype(np.float64)
    Lf = LSE.cpu().numpy().astype(np.float64)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(Of, Lf, O_ref, LSE_ref)
    # the same values through the contiguous entry point: identical bits
    Oc, Lc = pkg.attn_fwd(to_device(x["Q"]), to_device(x["K"]), to_device(x["V"]), scale=x["scale"], causal=causal,
                          key_padding_lens=lt)
    pkg.status_sync()
    assert torch.equal(O.contiguous(), Oc) and torch.equal(LSE, Lc)


def test_padded_rows_leave_the_gaps_untouched():
    import torch
    pkg = _pkg()
    B, H, N, d, pad = 2, 2, 300, 128, 8
    x = custom(B, H, N, N, d, True, seed=21)
    Q, K, V = bshd_view(x["Q"]), to_device(x["K"]), bshd_view(x["V"])   # K contiguous, the rest BSHD
    big = torch.full((B, N, H, d + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    O = big[..., :d].transpose(1, 2)                                     # row stride H * (d + pad)
    LSE = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    pkg.attn_fwd_strided(Q, K, V, O, LSE, scale=x["scale"], causal=True)
    pkg.status_sync()
    assert torch.all(big[..., d:] == 7.0), "the padding between rows was written"
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], True, None)
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)


def test_strided_argument_errors():
    import ctypes
    pkg = _pkg()
    lib = pkg.load_library()
    good = (ctypes.c_int64 * 3)(2 * 256 * 64, 256 * 64, 64)

    def call(qs):
        return lib.attn_fwd_strided(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 2, 256, 256, 64, 0.125, 0, None,
                                    qs, good, good, good, None)
    assert call((ctypes.c_int64 * 3)(0, 64, 64)) == -8           # zero stride
    assert call((ctypes.c_int64 * 3)(4096, 60, 64)) == -8        # not a multiple of 8 elements
    assert call(None) == -1


# ------------------------------------------------------------------ packed sequences

VARLEN = [
    # H, d, causal, query lengths, key lengths
    (3, 128, True, [300, 1, 0, 517], [300, 700, 5, 517]),
    (2, 64, False, [128, 129, 77], [64, 1000, 129]),
    (2, 128, False, [40, 250], [0, 260]),                        # a sequence with no keys
    (1, 128, True, [600, 600], [200, 600]),                      # Nq > Nk: leading rows fully masked
]


def packed(lengths, H, d, seed, tid_shift):
    """Per-sequence generator data [1, H, n, d] packed into [total, H, d] codes."""
    parts = []
    for i, n in enumerate(lengths):
        w = dict(name="packed", B=1, H=H, Nq=max(n, 1), Nk=max(n, 1), d=d, causal=False, qk=("normal", 0.0, 1.0),
                 v=("normal", 0.0, 1.0), seed=seed + 17 * i + tid_shift, lens=None, plant=None, scale=1.0)
        x = gen.make_inputs(w)
        parts.append((x["Q"][0, :, :n], x["K"][0, :, :n], x["V"][0, :, :n]))
    return parts


@pytest.mark.parametrize("H,d,causal,lq,lk", VARLEN)
def test_varlen_matches_oracle_per_sequence(H, d, causal, lq, lk):
    import torch
    pkg = _pkg()
    qparts = packed(lq, H, d, seed=300, tid_shift=0)
    kparts = packed(lk, H, d, seed=300, tid_shift=1)
    Qs = [p[0] for p in qparts]                        # [H, n, d] codes
    Ks = [p[1] for p in kparts]
    Vs = [p[2] for p in kparts]
    cat = lambda parts: np.ascontiguousarray(np.concatenate([p.transpose(1, 0, 2) for p in parts], axis=0))  # noqa
    Qp, Kp, Vp = cat(Qs), cat(Ks), cat(Vs)             # [total, H, d]
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    scale = 1.0 / math.sqrt(d)
    Q, K, V = to_device(Qp), to_device(Kp), to_device(Vp)
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((H, int(cu_q[-1])), float("nan"), dtype=torch.float32, device="cuda")
    pkg.attn_fwd_varlen(Q, K, V, torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda(), max(lq), O, LSE,
                        scale=scale, causal=causal)
    pkg.status_sync()
    Of = O.float().cpu().numpy().astype(np.float64)
    Lf = LSE.cpu().numpy().astype(np.float64)
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        rows = slice(cu_q[b], cu_q[b + 1])
        O_ref = np.zeros((H, lq[b], d))
        LSE_ref = np.zeros((H, lq[b]))
        for h in range(H):
            O_ref[h], LSE_ref[h] = oracle.attention_head(oracle.bf16_to_f64(Qs[b][h]), oracle.bf16_to_f64(Ks[b][h]),
                                                         oracle.bf16_to_f64(Vs[b][h]), scale, causal)
        compare(Of[rows].transpose(1, 0, 2), Lf[:, rows], O_ref, LSE_ref)
        # the same sequence alone through the contiguous entry point: identical bits
        if lk[b] > 0:
            Ob, Lb = pkg.attn_fwd(to_device(Qs[b][None]), to_device(Ks[b][None]), to_device(Vs[b][None]),
                                  scale=scale, causal=causal)
            pkg.status_sync()
            assert np.array_equal(Ob[0].float().cpu().numpy().transpose(1, 0, 2), O[rows].float().cpu().numpy())
            assert np.array_equal(Lb[0].cpu().numpy(), LSE[:, rows].cpu().numpy())
    assert not np.isnan(Of).any() and not np.isnan(Lf).any(), "a packed row was left unwritten"


def test_varlen_argument_errors():
    pkg = _pkg()
    lib = pkg.load_library()
    f = lib.attn_fwd_varlen
    base = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000, 2, 2, 128, 256, 256, 128, 0.1, 0, None]

    def call(**kw):
        a = list(base)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return f(*a)
    assert call(a12=96) == -3
    assert call(a7=-1) == -2
    assert call(a13=0.0) == -8
    assert call(a5=None) == -1
    assert call(a0=0x10008) == -4
    assert call(a9=0) == 0          # no query rows: nothing to do
