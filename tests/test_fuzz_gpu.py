"""Seeded random shapes through the public entry points, each compared element by element
with the fp64 oracle under the tolerance of the other parity tests.

The other files choose their shapes; these draw them from a fixed seed (the same cases
on every run): tails of every length, Nq != Nk in both directions, no keys at all, key
padding with zero, partial and full lengths, d = 64 and 128, causal or not, and packed
sequences of random lengths.  A slip in the masking, the tile decode, the item order or
the choice between the one-tile and two-tile kernels that the chosen shapes happen to
miss has more chances to show here.  The last six cases (d = 64, 80-100 heads, at least
three query tiles) have enough pairs of query tiles to take the two-tile kernel on a
152-SM GPU; the rest take the one-tile kernel.
"""
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, run_cuda, to_device

pytestmark = pytest.mark.gpu

SEED = 20261202


def _draw_fwd(n_small: int, n_many_heads: int):
    rng = np.random.default_rng(SEED)
    cases = []
    for i in range(n_small + n_many_heads):
        many = i >= n_small
        d = 64 if many else int(rng.choice([64, 128]))
        B = int(rng.integers(1, 3)) if many else int(rng.integers(1, 4))
        H = int(rng.integers(80, 101)) if many else int(rng.integers(1, 5))
        pick = rng.random()
        if many:
            Nq = int(rng.integers(257, 700))                 # >= 3 tiles: >= 160 pairs of tiles
        elif pick < 0.15:
            Nq = int(rng.integers(1, 6)) * 128              # whole tiles
        else:
            Nq = int(rng.integers(1, 700))
        pick = rng.random()
        if pick < 0.1 and not many:
            Nk = 0                                           # no keys: every row fully masked
        elif pick < 0.4:
            Nk = Nq
        else:
            Nk = int(rng.integers(1, 900))
        causal = bool(rng.random() < 0.5)
        lens = None
        if Nk > 0 and rng.random() < 0.4:
            lens = [int(v) for v in rng.integers(0, Nk + 1, size=B)]
            if B > 1 and rng.random() < 0.5:
                lens[int(rng.integers(B))] = 0               # a batch with no visible key
            if rng.random() < 0.5:
                lens[int(rng.integers(B))] = Nk
        cases.append((i, B, H, Nq, Nk, d, causal, lens))
    return cases


FWD_CASES = _draw_fwd(30, 6)


@pytest.mark.parametrize("i,B,H,Nq,Nk,d,causal,lens", FWD_CASES,
                         ids=[f"c{c[0]}-B{c[1]}H{c[2]}q{c[3]}k{c[4]}d{c[5]}{'c' if c[6] else 'n'}"
                              f"{'' if c[7] is None else 'L'}" for c in FWD_CASES])
def test_random_shape_matches_oracle(i, B, H, Nq, Nk, d, causal, lens):
    w = dict(name="fuzz", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=SEED + 101 * i, lens=None if lens is None else ("given", lens),
             plant=None, scale=1.0 / math.sqrt(d))
    x = gen.make_inputs(w)
    O, LSE = run_cuda(x)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], x["causal"], x["lens"])
    compare(O, LSE, O_ref, LSE_ref)


def _draw_varlen(n: int):
    rng = np.random.default_rng(SEED + 1)
    cases = []
    for i in range(n):
        nseq = int(rng.integers(1, 7))
        lq = [int(v) for v in rng.integers(0, 600, size=nseq)]
        lk = [q if rng.random() < 0.4 else int(v) for q, v in zip(lq, rng.integers(0, 700, size=nseq))]
        cases.append((i, int(rng.integers(1, 4)), int(rng.choice([64, 128])), bool(rng.random() < 0.5), lq, lk))
    return cases


VARLEN_CASES = _draw_varlen(10)


def _sequence(n, H, d, seed):
    """[H, n, d] codes of one sequence (n may be 0)."""
    w = dict(name="fuzz_seq", B=1, H=H, Nq=max(n, 1), Nk=max(n, 1), d=d, causal=False, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None, plant=None, scale=1.0)
    x = gen.make_inputs(w)
    return x["Q"][0, :, :n], x["K"][0, :, :n], x["V"][0, :, :n]


@pytest.mark.parametrize("i,H,d,causal,lq,lk", VARLEN_CASES, ids=[f"v{c[0]}" for c in VARLEN_CASES])
def test_random_packed_sequences_match_oracle(i, H, d, causal, lq, lk):
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    qs = [_sequence(n, H, d, SEED + 1000 * i + 2 * b)[0] for b, n in enumerate(lq)]
    kv = [_sequence(n, H, d, SEED + 1000 * i + 2 * b + 1) for b, n in enumerate(lk)]
    ks, vs = [t[1] for t in kv], [t[2] for t in kv]
    cat = lambda parts: np.ascontiguousarray(np.concatenate([p.transpose(1, 0, 2) for p in parts], axis=0))  # noqa: E731
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    if cu_q[-1] == 0:
        pytest.skip("the draw has no query rows")
    scale = 1.0 / math.sqrt(d)
    Q, K, V = to_device(cat(qs)), to_device(cat(ks)), to_device(cat(vs))
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((H, int(cu_q[-1])), float("nan"), dtype=torch.float32, device="cuda")
    pkg.attn_fwd_varlen(Q, K, V, torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda(), max(lq), O, LSE,
                        scale=scale, causal=causal)
    pkg.status_sync()
    Of = O.float().cpu().numpy().astype(np.float64)
    Lf = LSE.cpu().numpy().astype(np.float64)
    assert not np.isnan(Of).any() and not np.isnan(Lf).any(), "a packed row was left unwritten"
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        rows = slice(cu_q[b], cu_q[b + 1])
        O_ref = np.zeros((H, lq[b], d))
        L_ref = np.zeros((H, lq[b]))
        for h in range(H):
            O_ref[h], L_ref[h] = oracle.attention_head(oracle.bf16_to_f64(qs[b][h]), oracle.bf16_to_f64(ks[b][h]),
                                                       oracle.bf16_to_f64(vs[b][h]), scale, causal)
        compare(Of[rows].transpose(1, 0, 2), Lf[:, rows], O_ref, L_ref)


def _draw_layouts(n: int):
    """Strided problems: every tensor stored [B, N, H', d'] with H' >= H heads and d' >= d
    columns per row (gaps between heads and between rows), viewed as [B, H, N, d]."""
    rng = np.random.default_rng(SEED + 2)
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        B, H = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        Nq, Nk = int(rng.integers(1, 600)), int(rng.integers(1, 800))
        causal = bool(rng.random() < 0.5)
        lens = [int(v) for v in rng.integers(0, Nk + 1, size=B)] if rng.random() < 0.3 else None
        extra_h = int(rng.integers(0, 3))                     # unused heads between the used ones
        extra_d = int(rng.choice([0, 8, 64]))                 # unused columns after each row
        cases.append((i, B, H, Nq, Nk, d, causal, lens, extra_h, extra_d))
    return cases


LAYOUT_CASES = _draw_layouts(12)


def _strided(codes, extra_h, extra_d, fill):
    """[B, H, N, d] codes placed in a [B, N, H + extra_h, d + extra_d] tensor, returned as
    the [B, H, N, d] view and the whole storage."""
    import torch
    B, H, N, d = codes.shape
    big = torch.full((B, N, H + extra_h, d + extra_d), fill, dtype=torch.bfloat16, device="cuda")
    view = big[:, :, :H, :d].transpose(1, 2)
    view.copy_(to_device(codes))
    return view, big


@pytest.mark.parametrize("i,B,H,Nq,Nk,d,causal,lens,extra_h,extra_d", LAYOUT_CASES,
                         ids=[f"s{c[0]}" for c in LAYOUT_CASES])
def test_random_strided_layouts_match_oracle(i, B, H, Nq, Nk, d, causal, lens, extra_h, extra_d):
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    w = dict(name="fuzz_strided", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=SEED + 303 * i, lens=None if lens is None else ("given", lens),
             plant=None, scale=1.0 / math.sqrt(d))
    x = gen.make_inputs(w)
    Q, _ = _strided(x["Q"], extra_h, extra_d, 0.0)
    K, _ = _strided(x["K"], extra_h, extra_d, 0.0)
    V, _ = _strided(x["V"], extra_h, extra_d, 0.0)
    O, Obig = _strided(np.zeros((B, H, Nq, d), np.uint16), extra_h, extra_d, 7.0)
    LSE = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    lt = None if lens is None else torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    pkg.attn_fwd_strided(Q, K, V, O, LSE, scale=x["scale"], causal=causal, key_padding_lens=lt)
    pkg.status_sync()
    if extra_d:
        assert torch.all(Obig[..., d:] == 7.0), "the gap after a row of O was written"
    if extra_h:
        assert torch.all(Obig[:, :, H:, :] == 7.0), "an unused head of O was written"
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)


def _draw_splitkv(n: int):
    """Few query rows against long key ranges, the shapes split-KV is for."""
    rng = np.random.default_rng(SEED + 3)
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 5))
        Nq, Nk = int(rng.integers(1, 300)), int(rng.integers(200, 5000))
        causal = bool(rng.random() < 0.5)
        lens = [int(v) for v in rng.integers(0, Nk + 1, size=B)] if rng.random() < 0.4 else None
        splits = int(rng.choice([0, 2, 3, 5, 8]))            # 0: the library chooses
        cases.append((i, B, H, Nq, Nk, d, causal, lens, splits))
    return cases


SPLITKV_FUZZ = _draw_splitkv(10)


@pytest.mark.parametrize("i,B,H,Nq,Nk,d,causal,lens,splits", SPLITKV_FUZZ, ids=[f"k{c[0]}" for c in SPLITKV_FUZZ])
def test_random_splitkv_matches_oracle(i, B, H, Nq, Nk, d, causal, lens, splits):
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    w = dict(name="fuzz_splitkv", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=SEED + 505 * i, lens=None if lens is None else ("given", lens),
             plant=None, scale=1.0 / math.sqrt(d))
    x = gen.make_inputs(w)
    lt = None if lens is None else torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    O, LSE = pkg.attn_fwd_splitkv(to_device(x["Q"]), to_device(x["K"]), to_device(x["V"]), num_splits=splits,
                                  scale=x["scale"], causal=causal, key_padding_lens=lt)
    pkg.status_sync()
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)
