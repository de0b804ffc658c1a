"""Split-KV on the GPU, through the C ABI, against the fp64 oracle.

* attn_fwd_states: every split's state (m, l, o~) element by element against the
  oracle's state over the same key range (the ranges follow the rule the header
  states), including splits that hold no visible key.
* attn_merge_states: the merge kernel alone on states the oracle wrote, including
  maxima a thousand apart and rows whose states are all empty.
* attn_fwd_splitkv: the merged result against the three-pass oracle, for explicit and
  automatic split counts, and at full size on sampled rows of the decoding shape.

Tolerance: the states' o~ / l and the merged O follow the forward's O bound
(|dO| <= 1e-2 s_V + half a bf16 ulp where O is bf16), m and LSE within 1e-3, and
l within a relative 1e-3 (the same bound as LSE, read on l = exp(LSE - m)).
"""
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import ATOL_LSE, ATOL_O, compare, run_cuda, sample_rows, to_device

pytestmark = pytest.mark.gpu


def _pkg():
    import online_softmax_flashattention_attention_gb300 as pkg
    return pkg


def _problem(B, H, Nq, Nk, d, causal, seed, lens=None, sigma=1.0):
    w = dict(name="splitkv", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, sigma),
             v=("normal", 0.0, 1.0), seed=seed, lens=None if lens is None else ("given", lens), plant=None,
             scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def split_ranges(Nk, S):
    """Split s covers keys [s*C, (s+1)*C) within [0, Nk), C = 128 * ceil(ceil(Nk/128) / S)."""
    nkb = -(-Nk // 128)
    C = 128 * max(1, -(-nkb // S))
    return [(min(s * C, Nk), min((s + 1) * C, Nk)) for s in range(S)]


def _lens_dev(x):
    import torch
    return None if x["lens"] is None else torch.as_tensor(np.asarray(x["lens"], np.int32)).cuda()


STATE_CASES = [
    # B, H, Nq, Nk, d, causal, lens, S
    (2, 3, 300, 700, 128, True, [700, 333], 3),
    (1, 2, 200, 520, 64, False, None, 5),
    (1, 2, 130, 256, 128, False, None, 4),       # splits 2 and 3 hold no key at all
    (2, 1, 64, 1000, 128, True, [0, 1000], 2),   # batch 0 fully masked
]


@pytest.mark.parametrize("case", STATE_CASES)
def test_states_match_oracle_states(case):
    B, H, Nq, Nk, d, causal, lens, S = case
    pkg = _pkg()
    x = _problem(B, H, Nq, Nk, d, causal, seed=60 + S, lens=lens)
    o, m, l = pkg.attn_fwd_states(to_device(x["Q"]), to_device(x["K"]), to_device(x["V"]), S, scale=x["scale"],
                                  causal=causal, key_padding_lens=_lens_dev(x))
    pkg.status_sync()
    o, m, l = (t.cpu().numpy().astype(np.float64) for t in (o, m, l))
    ro, rm, rl = oracle.attention_states(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"],
                                         split_ranges(Nk, S))
    empty = np.isneginf(rm)
    assert np.array_equal(np.isneginf(m), empty), "empty states differ"
    assert np.all(l[empty] == 0.0) and np.all(o[empty] == 0.0)
    live = ~empty
    assert np.abs(m[live] - rm[live]).max() <= ATOL_LSE
    assert np.abs(l[live] / rl[live] - 1.0).max() <= ATOL_LSE
    err = np.abs(o[live] / l[live][:, None] - ro[live] / rl[live][:, None])
    assert err.max() <= ATOL_O, err.max()


def _oracle_states_f32(rng, S, rows, d):
    """States the oracle computed over random key sets, rounded to fp32, with maxima
    far apart and some empty ones."""
    o = np.zeros((S, rows, d))
    m = np.full((S, rows), -np.inf)
    l = np.zeros((S, rows))
    for s in range(S):
        n = 200                                         # scores with a spread of 1 to 3
        q = rng.normal(size=(rows, 16))
        k = rng.normal(size=(n, 16)) * (1 + s % 3)
        v = rng.normal(size=(n, d))
        o[s], m[s], l[s] = oracle.attention_state_head(q, k, v, 0.25, False, None, 0, n)
        m[s] += 1000.0 * (s % 2)                      # shift: the same state, reference moved
    m[:, :5] = -np.inf                                  # rows 0..4: every state empty
    l[:, :5] = 0.0
    o[:, :5] = 0.0
    if S > 1:                                           # rows 5..8: one empty state
        m[1, 5:9] = -np.inf
        l[1, 5:9] = 0.0
        o[1, 5:9] = 0.0
    return o.astype(np.float32), m.astype(np.float32), l.astype(np.float32)


@pytest.mark.parametrize("S,rows,d", [(1, 37, 128), (3, 300, 128), (7, 129, 64), (40, 70, 128)])
def test_merge_kernel_matches_oracle_merge(S, rows, d):
    import torch
    pkg = _pkg()
    rng = np.random.default_rng(100 + S)
    o, m, l = _oracle_states_f32(rng, S, rows, d)
    O, LSE = pkg.merge_states(torch.from_numpy(o).cuda(), torch.from_numpy(m).cuda(), torch.from_numpy(l).cuda())
    torch.cuda.synchronize()
    ro, rm, rl = oracle.merge_states([(o[s].astype(np.float64), m[s].astype(np.float64), l[s].astype(np.float64))
                                      for s in range(S)])
    O_ref, LSE_ref = oracle.finish_state(ro, rm, rl)
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)
    assert np.all(np.isneginf(LSE.cpu().numpy()[:5])) and not O.float().cpu().numpy()[:5].any()


SPLITKV_CASES = [
    (2, 3, 300, 700, 128, True, [700, 333], 3),
    (1, 2, 200, 520, 64, False, None, 5),
    (1, 4, 128, 4096, 128, True, None, 0),          # automatic split count
    (1, 2, 100, 3000, 64, True, [2000], 0),
    (2, 1, 64, 1000, 128, False, [0, 1000], 2),
    (1, 1, 16, 0, 128, False, None, 3),             # no keys at all
]


@pytest.mark.parametrize("case", SPLITKV_CASES)
def test_splitkv_matches_oracle(case):
    import torch
    B, H, Nq, Nk, d, causal, lens, S = case
    pkg = _pkg()
    x = _problem(B, H, Nq, Nk, d, causal, seed=80 + S, lens=lens)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    pkg.attn_fwd_splitkv(Q, K, V, O, LSE, num_splits=S, scale=x["scale"], causal=causal,
                         key_padding_lens=_lens_dev(x))
    pkg.status_sync()
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)
    if Nk > 0:  # and it agrees with the one-pass kernel within the same bound
        O1, LSE1 = run_cuda(x)
        assert np.abs(O.float().cpu().numpy() - O1).max() <= 2 * ATOL_O


def test_automatic_split_count_fills_the_sms():
    import torch
    pkg = _pkg()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert pkg.splitkv_splits(1, 32, 128, 32768) == sms // 32
    assert pkg.splitkv_splits(2, 32, 8192, 8192) == 1       # 4096 tiles already fill the SMs
    assert pkg.splitkv_splits(1, 1, 128, 256) == 1          # too few key blocks to split


def test_splitkv_full_size_decode_shape_sampled_rows():
    import torch
    pkg = _pkg()
    x = gen.make_inputs("causal_b1h32q128k32768d128")
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    S = pkg.splitkv_splits(1, 32, 128, 32768)
    O, LSE = pkg.attn_fwd_splitkv(Q, K, V, num_splits=S, scale=x["scale"], causal=True)
    pkg.status_sync()
    picks = sample_rows(1, 32, 128, n_random=24, seed=5)
    O_ref, LSE_ref = oracle.attention_rows(x["Q"], x["K"], x["V"], x["scale"], True, None, picks)
    Of = O.float().cpu().numpy()
    Lf = LSE.cpu().numpy()
    got_O = np.stack([Of[b, h, i] for b, h, i in picks]).astype(np.float64)
    got_L = np.array([Lf[b, h, i] for b, h, i in picks], dtype=np.float64)
    compare(got_O, got_L, O_ref, LSE_ref)
