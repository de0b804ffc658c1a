"""attn_fwd_ex options on the GPU against the fp64 oracle: every exponential on the MUFU
unit, the mixed (polynomial + MUFU) default, and the lazy rescale threshold.

The lazy rescale changes only the reference point of the running sums; softmax is
invariant to it ("FlashAttention math", "Safe softmax"), so every variant must meet the
same tolerance as attn_fwd.  The cases include maxima that rise block after block by
more than the threshold, planted large scores and scores far beyond the float32 exp
range, a row with a single visible key (exact), and padding against truncation.
"""
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, to_device

pytestmark = pytest.mark.gpu

MODES = [  # (rescale_threshold, exp2_mode)
    (0.0, 1),    # the pages' rescale rule, ex2.approx only
    (0.0, 2),    # the pages' rule, mixed exponentials
    (5.5, 2),    # lazy rescale (factor ~2^8)
    (20.0, 1),   # the largest threshold allowed
]


def _pkg():
    import online_softmax_flashattention_attention_gb300 as pkg
    return pkg


def custom(B, H, Nq, Nk, d, causal=False, seed=7, lens=None, qk=("normal", 0.0, 1.0), v=("normal", 0.0, 1.0)):
    w = dict(name="custom", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=qk, v=v, seed=seed,
             lens=None if lens is None else ("given", lens), plant=None, scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def run_ex(x, tau, mode, Q=None, K=None, V=None, lens=None, Nk=None, key_block=0):
    import torch
    pkg = _pkg()
    Q = to_device(x["Q"]) if Q is None else Q
    K = to_device(x["K"]) if K is None else K
    V = to_device(x["V"]) if V is None else V
    B, H, Nq, d = Q.shape
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    lens = x["lens"] if lens is None else lens
    lt = None if lens is None else torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    pkg.attn_fwd(Q, K, V, O, LSE, scale=x["scale"], causal=x["causal"], key_padding_lens=lt,
                 rescale_threshold=tau, exp2_mode=mode, key_block=key_block)
    pkg.status_sync()
    return O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64)


SHAPES = [
    (2, 3, 300, 300, 128, True, None),
    (2, 2, 300, 512, 64, True, [512, 127]),
    (3, 1, 260, 700, 128, False, [0, 1, 700]),
    (1, 2, 640, 640, 64, False, None),
]


@pytest.mark.parametrize("tau,mode", MODES)
@pytest.mark.parametrize("shape", SHAPES)
def test_modes_match_oracle(shape, tau, mode):
    B, H, Nq, Nk, d, causal, lens = shape
    x = custom(B, H, Nq, Nk, d, causal, seed=Nq + Nk + d, lens=lens)
    O, LSE = run_ex(x, tau, mode)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O, LSE, O_ref, LSE_ref)


def rising_max_problem(d=128, Nk=1024, step=12.0):
    """One query whose score with key j is step * (j // 128): the max rises by `step`
    natural-log units every block, so with threshold 5.5 every block rescales and with
    threshold 20 every other block does (p then reaches exp(12) within a block)."""
    import torch
    q = np.zeros((1, 1, 1, d), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, Nk, d), np.float32)
    k[0, 0, :, 0] = step * (np.arange(Nk) // 128)
    rng = np.random.default_rng(3)
    v = rng.normal(size=(1, 1, Nk, d)).astype(np.float32)
    to = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()  # noqa: E731
    Qt, Kt, Vt = to(q), to(k), to(v)
    # the oracle reads the same bf16 values
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    return Qt, Kt, Vt, f(Qt), f(Kt), f(Vt)


@pytest.mark.parametrize("tau,mode", MODES)
def test_max_rising_every_block(tau, mode):
    Qt, Kt, Vt, q, k, v = rising_max_problem()
    x = dict(scale=1.0, causal=False, lens=None)
    O, LSE = run_ex(x, tau, mode, Q=Qt, K=Kt, V=Vt)
    O_ref, LSE_ref = oracle.attention(q, k, v, 1.0, False, None)
    compare(O, LSE, O_ref, LSE_ref)


@pytest.mark.parametrize("tau,mode", MODES)
def test_huge_scores_stay_finite(tau, mode):
    # scores with a spread of ~30: the largest pass 88, where float32 exp overflows unshifted
    x = custom(1, 2, 256, 512, 128, False, seed=11, qk=("normal", 0.0, 5.5))
    O, LSE = run_ex(x, tau, mode)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(LSE))
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    compare(O, LSE, O_ref, LSE_ref)


@pytest.mark.parametrize("tau,mode", MODES)
def test_single_visible_key_exact(tau, mode):
    # causal with Nq = Nk: row 0 sees key 0 only, so O[0] = V[0] exactly
    x = custom(1, 2, 200, 200, 128, True, seed=12)
    O, LSE = run_ex(x, tau, mode)
    V = gen.codes_to_f32(x["V"]).astype(np.float64)
    assert np.array_equal(O[:, :, 0], V[:, :, 0])


@pytest.mark.parametrize("tau,mode", MODES)
def test_padding_equals_truncation_bitwise(tau, mode):
    import torch
    x = custom(2, 2, 256, 640, 64, False, seed=13, lens=[640, 300])
    O, LSE = run_ex(x, tau, mode)
    # batch 1 alone with its keys cut to 300
    xb = dict(scale=x["scale"], causal=False, lens=None)
    Q1 = to_device(x["Q"][1:2])
    K1 = to_device(np.ascontiguousarray(x["K"][1:2, :, :300]))
    V1 = to_device(np.ascontiguousarray(x["V"][1:2, :, :300]))
    O1, LSE1 = run_ex(xb, tau, mode, Q=Q1, K=K1, V=V1)
    assert np.array_equal(O[1:2], O1) and np.array_equal(LSE[1:2], LSE1)
    del torch


def test_mixed_and_hardware_exponentials_agree_closely():
    x = custom(2, 4, 512, 512, 128, True, seed=14)
    Oh, Lh = run_ex(x, 0.0, 1)
    Om, Lm = run_ex(x, 0.0, 2)
    # the polynomial's relative error (< 3e-6) is far below the bf16 rounding of P and O
    assert np.abs(Oh - Om).max() <= 2.0 ** -7
    assert np.abs(Lh - Lm).max() <= 1e-4


def test_planted_workload_lazy_sampled_rows():
    # scores ~60 in the first or the last valid tile, V in [-100, 100], one fully masked batch
    x = gen.make_inputs("padded_planted_b2h8n4096d128")
    O, LSE = run_ex(x, 5.5, 2)
    assert np.all(O[0] == 0) and np.all(np.isneginf(LSE[0]))
    from gpu_helpers import sample_rows
    picks = sample_rows(2, 8, 4096, n_random=24, seed=9)
    O_ref, LSE_ref = oracle.attention_rows(x["Q"], x["K"], x["V"], x["scale"], False, x["lens"], picks)
    idx = tuple(np.array(picks).T)
    compare(O[idx], LSE[idx], O_ref, LSE_ref, s_v=100.0)


def test_largest_threshold_with_values_of_100():
    """tau = 20, the largest threshold allowed, with the max rising by 19.5 (just under tau)
    every other block, so that p reaches e^19.5 ~ 2.9e8 before the reference moves, and V
    uniform in [-100, 100]: |o~| reaches ~4e12, far inside the stated bound
    Nk e^tau max|V| < FLT_MAX, and the result must meet the s_V = 100 tolerance."""
    import torch
    Qt, Kt, _, q, k, _ = rising_max_problem(step=19.5)
    rng = np.random.default_rng(21)
    Vt = torch.from_numpy(rng.uniform(-100.0, 100.0, size=(1, 1, Kt.shape[2], Kt.shape[3])).astype(np.float32)
                          ).to(torch.bfloat16).cuda()
    v = Vt.float().cpu().numpy().astype(np.float64)
    x = dict(scale=1.0, causal=False, lens=None)
    for mode in (1, 2):
        O, LSE = run_ex(x, 20.0, mode, Q=Qt, K=Kt, V=Vt)
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(LSE))
        O_ref, LSE_ref = oracle.attention(q, k, v, 1.0, False, None)
        compare(O, LSE, O_ref, LSE_ref, s_v=100.0)


# ------------------------------------------------------------------ key-block size

WIDE_SHAPES = [
    (2, 3, 300, 300, True, None),
    (3, 1, 260, 700, False, [0, 1, 700]),
    (1, 2, 200, 383, True, None),             # Nq < Nk, bottom-right causal
    (1, 2, 383, 200, True, None),             # Nq > Nk: first rows fully masked
    (2, 2, 640, 1000, False, [1000, 191]),    # padding inside the first and the sixth block
    (2, 40, 300, 600, True, None),            # more items than SMs
]


@pytest.mark.parametrize("kb", [64, 192])
@pytest.mark.parametrize("shape", WIDE_SHAPES)
def test_key_block_matches_128_and_oracle(shape, kb):
    """The recurrence's result does not depend on the key-block size ("FlashAttention
    math", "Proof of exactness"; "Tiled attention: running max softmax" varies the tile):
    the 64- and 192-key builds agree with the oracle and with the 128-key build within
    the tolerance, with the pages' rescale rule and with the lazy option."""
    B, H, Nq, Nk, causal, lens = shape
    x = custom(B, H, Nq, Nk, 128, causal, seed=Nq + Nk + 5, lens=lens)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    for tau in (0.0, 5.5):
        O128, L128 = run_ex(x, tau, 1)
        Okb, Lkb = run_ex(x, tau, 1, key_block=kb)
        compare(Okb, Lkb, O_ref, LSE_ref)
        compare(Okb, Lkb, O128, L128)


@pytest.mark.parametrize("kb", [64, 192])
def test_key_block_full_size_every_item(kb):
    """B4 H16 N2048 d128 causal with 64- or 192-key blocks: two rows of every work item
    against the oracle, and every row against the 128-key build."""
    x = gen.make_inputs("causal_b4h16n2048d128")
    Okb, Lkb = run_ex(x, 0.0, 1, key_block=kb)
    O128, L128 = run_ex(x, 0.0, 1)
    compare(Okb, Lkb, O128, L128)
    rng = np.random.default_rng(12)
    picks = sorted({p for b in range(4) for h in range(16) for t0 in range(0, 2048, 128)
                    for p in ((b, h, int(rng.integers(t0, t0 + 128))), (b, h, t0 + 127))})
    O_ref, LSE_ref = oracle.attention_rows(x["Q"], x["K"], x["V"], x["scale"], True, None, picks)
    idx = tuple(np.array(picks).T)
    compare(Okb[idx], Lkb[idx], O_ref, LSE_ref)


@pytest.mark.parametrize("kb", [64, 192])
def test_key_block_rejected_where_not_built(kb):
    pkg = _pkg()
    x = custom(1, 2, 256, 256, 64, False, seed=3)
    with pytest.raises(pkg.AttnError) as err:
        run_ex(x, 0.0, 1, key_block=kb)           # d = 64
    assert err.value.status == -8
    x = custom(1, 2, 256, 256, 128, False, seed=4)
    with pytest.raises(pkg.AttnError) as err:
        run_ex(x, 0.0, 2, key_block=kb)           # mixed exponentials
    assert err.value.status == -8
    with pytest.raises(pkg.AttnError) as err:
        run_ex(x, 0.0, 1, key_block=96)           # a size that is not built
    assert err.value.status == -8
