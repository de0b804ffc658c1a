"""Pins of the fp64 oracle to things other than itself.

Each test checks the oracle against the pages' printed worked examples
(tests/golden/page_examples.json, cited per entry), closed forms, invariants
the pages prove, an independent library routine (scipy's logsumexp) or brute
force on tiny inputs with the unshifted definition.  The mutation tests plant
the pages' own list of mistakes in the oracle's blockwise recurrence and check
that a pin catches each one.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def one_dim_problem(scores, V):
    """q = [1], k_j = [s_j], scale 1: the oracle's scores are exactly the given ones."""
    s = np.asarray(scores, dtype=np.float64)
    q = np.ones((1, 1))
    k = s[:, None]
    v = np.asarray(V, dtype=np.float64)
    if v.ndim == 1:
        v = v[:, None]
    return q, k, v


# ---------------------------------------------------------------- page examples

def test_softmax_2413_printed(golden):
    g = golden["softmax_2413"]
    s = np.array(g["scores"], dtype=float)
    assert np.allclose(np.exp(s), g["numerators"], atol=g["numerators_tol"])
    assert abs(np.exp(s).sum() - g["denominator"]) <= g["denominator_tol"]
    for f in (oracle.softmax_naive, oracle.softmax_safe):
        assert np.allclose(f(s), g["softmax"], atol=g["tol"], rtol=0)


def test_safe_2413_m_and_l(golden):
    g = golden["safe_2413"]
    m, l = oracle.softmax_stats(g["scores"])
    assert m == g["m"]
    assert abs(l - g["l"]) <= g["tol"]
    assert np.allclose(np.exp(np.array(g["scores"]) - m), g["shifted_numerators"], atol=g["tol"])
    # m and l are all you need: e^{s_i - m} / l is the softmax
    assert np.allclose(np.exp(np.array(g["scores"]) - m) / l, golden["softmax_2413"]["softmax"], atol=5e-4)


def test_large_scores_and_overflow(golden):
    g = golden["large_scores"]
    s = np.array(g["scores"], dtype=float)
    assert np.allclose(np.exp(s), g["exp"], rtol=g["exp_rtol"])
    # naive softmax still works here (exp(102) is finite in float64) ...
    assert np.allclose(oracle.softmax_naive(s), oracle.softmax_safe(s), rtol=1e-12)
    # ... but breaks at the float64 overflow point while the safe path does not
    big = s + g["float64_exp_overflows_at"]
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(float(g["float64_exp_overflows_at"])))
    assert not np.all(np.isfinite(oracle.softmax_naive(big)))
    safe = oracle.softmax_safe(big)
    assert np.all(np.isfinite(safe)) and np.allclose(safe, oracle.softmax_safe(s), rtol=1e-12)


def test_float32_overflow_point(golden):
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(np.float32(golden["float32_overflow"]["score_that_overflows_float32"])))
        assert np.isfinite(np.exp(np.float32(88.0)))


def test_block_trace_2413(golden):
    g = golden["blocks_2413"]
    s = np.array(sum(g["blocks"], []), dtype=float)
    tr = []
    o, m, l = oracle.online_softmax_attention(s, np.zeros(4), block=2, trace=tr)
    for st, want in zip(tr, g["after"]):
        assert st["m"] == want["m"] and abs(st["l"] - want["l"]) <= g["tol"]
    # each block against its own max, summed: the page's wrong total (with its
    # exp(1-3) slip corrected; see "slip" in the fixture)
    local = [oracle.softmax_stats(b)[1] for b in g["blocks"]]
    assert np.allclose(local, g["naive_local_l_reading"], atol=g["tol"])
    assert abs(sum(local) - g["naive_wrong_sum_reading"]) <= g["tol"]
    assert abs(local[1] - g["naive_local_l_printed"][1]) > 0.2   # the printed slip itself
    assert abs(sum(local) - g["after"][-1]["l"]) > 0.5 and abs(g["naive_wrong_sum_printed"] - g["after"][-1]["l"]) > 0.5


def test_block_trace_1253(golden):
    g = golden["blocks_1253"]
    s = np.array(sum(g["blocks"], []), dtype=float)
    tr = []
    oracle.online_softmax_attention(s, np.zeros(4), block=2, trace=tr)
    for st, want in zip(tr, g["after"]):
        assert st["m"] == want["m"] and abs(st["l"] - want["l"]) <= g["tol"]
    assert abs(tr[1]["alpha"] - g["scale"]) <= g["tol"]
    assert abs(tr[0]["l"] * tr[1]["alpha"] - g["rescaled_l"]) <= g["tol"]


@pytest.mark.parametrize("key", ["attention_no_rescale", "attention_rescale"])
def test_attention_two_blocks(golden, key):
    g = golden[key]
    s = np.array(g["scores"], dtype=float)
    V = np.array(g["V"], dtype=float)
    tol = g["tol"]
    tol_r = g.get("tol_rounded", tol)
    tr = []
    out, m, l = oracle.online_softmax_attention(s, V, block=g["block"], trace=tr)
    for st, want in zip(tr, g["after"]):
        assert st["m"] == want["m"]
        assert abs(st["l"] - want["l"]) <= tol
        assert np.allclose(st["o"], want["o"], atol=tol)
    if "rescale" in g:
        r = g["rescale"]
        assert abs(tr[1]["alpha"] - r["scale"]) <= tol
        assert abs(tr[0]["l"] * tr[1]["alpha"] - r["l"]) <= tol
        assert np.allclose(tr[0]["o"] * tr[1]["alpha"], r["o"], atol=tol)
    # the oracle proper (three-pass, matmul) on the same problem
    q, k, v = one_dim_problem(s, V)
    O, LSE = oracle.attention_head(q, k, v, scale=1.0)
    for want in [g["output"]] + ([g["output_verification"]] if "output_verification" in g else []):
        assert np.allclose(O[0], want, atol=tol_r)
        assert np.allclose(out, want, atol=tol_r)
    assert np.allclose(oracle.softmax_safe(s), g["P"], atol=tol_r)
    # V = identity turns the output into the probabilities themselves
    O_eye, _ = oracle.attention_head(q, k, np.eye(4), scale=1.0)
    assert np.allclose(O_eye[0], g["P"], atol=tol_r)
    assert abs(LSE[0] - (m + math.log(l))) < 1e-12


def test_scalar_values_example(golden):
    g = golden["scalar_values"]
    s = np.array(g["scores"], dtype=float)
    v = np.array(g["v"], dtype=float)
    m, l = oracle.softmax_stats(s)
    assert np.allclose(np.exp(s - m), g["weights"], atol=g["tol"])
    assert abs(l - g["l"]) <= g["tol"]
    assert abs(np.exp(s - m) @ v - g["o_tilde"]) <= 5e-4
    tr = []
    o, m2, l2 = oracle.online_softmax_attention(s, v, block=g["block"], trace=tr)
    assert abs(o - g["o"]) <= g["tol_o"]
    for st, want in zip(tr, g["blocks"]):
        assert st["m_blk"] == want["m_blk"] and st["m"] == want["m"]
        assert abs(st["alpha"] - want["alpha"]) <= g["tol"]
        assert np.allclose(st["p"], want["p"], atol=g["tol"])
        assert abs(st["l"] - want["l"]) <= g["tol"]
        assert abs(st["o"][0] - want["o"]) <= 5e-4
    q, k, vv = one_dim_problem(s, v)
    O, LSE = oracle.attention_head(q, k, vv, scale=1.0)
    assert abs(O[0, 0] - g["o"]) <= g["tol_o"]
    assert abs(LSE[0] - logsumexp(s)) < 1e-12


def test_quiz_rescale_factor(golden):
    g = golden["quiz_rescale_factor"]
    scale = math.exp(g["m_old"] - max(g["m_old"], g["m_block"]))
    assert abs(scale - g["scale"]) <= g["tol"]
    assert abs(g["l_old"] * scale - g["l_new"]) <= g["tol"]


def test_quiz_three_blocks(golden):
    g = golden["quiz_three_blocks"]
    tr = []
    oracle.online_softmax_attention(g["scores"], np.ones(3), block=1, trace=tr)
    assert [t["m"] for t in tr] == g["m"]
    assert np.allclose([t["alpha"] for t in tr], g["scale"], atol=g["tol"])


def test_quiz_rescale_l_only_factor(golden):
    g = golden["quiz_rescale_l_only"]
    factor = 1.0 / math.exp(g["m_old"] - g["m_new"])
    assert abs(factor - g["too_large_factor"]) / g["too_large_factor"] <= 0.01 + 0.005


# ---------------------------------------------------------------- brute force

def brute_force(Q, K, V, scale, causal=False, key_len=None):
    """Unshifted definition with explicit loops (tiny inputs, |s| well below 709)."""
    Nq, d = Q.shape
    Nk = K.shape[0]
    dv = V.shape[1]
    O = [[0.0] * dv for _ in range(Nq)]
    LSE = [-math.inf] * Nq
    L = Nk if key_len is None else min(max(key_len, 0), Nk)
    for i in range(Nq):
        w = []
        for j in range(Nk):
            ok = j < L and (not causal or j <= i + (Nk - Nq))
            if ok:
                sc = scale * sum(float(Q[i, t]) * float(K[j, t]) for t in range(d))
                w.append((j, math.exp(sc)))
        tot = sum(x for _, x in w)
        if tot > 0:
            for c in range(dv):
                O[i][c] = sum(x * float(V[j, c]) for j, x in w) / tot
            LSE[i] = math.log(tot)
    return np.array(O), np.array(LSE)


@pytest.mark.parametrize("Nq,Nk,d,dv,causal,key_len", [
    (5, 7, 3, 4, False, None), (7, 5, 3, 2, True, None), (6, 6, 4, 4, True, None),
    (4, 9, 2, 3, False, 6), (9, 4, 3, 3, True, 3), (3, 8, 5, 1, True, 0), (8, 3, 2, 2, True, None),
])
def test_oracle_vs_brute_force(Nq, Nk, d, dv, causal, key_len):
    rng = np.random.default_rng(Nq * 100 + Nk * 10 + d)
    Q, K, V = rng.normal(size=(Nq, d)), rng.normal(size=(Nk, d)), rng.normal(size=(Nk, dv))
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.attention_head(Q, K, V, scale, causal, key_len)
    Ob, LSEb = brute_force(Q, K, V, scale, causal, key_len)
    assert np.allclose(O, Ob, rtol=1e-12, atol=1e-13)
    live = np.isfinite(LSEb)
    assert np.array_equal(live, np.isfinite(LSE))
    assert np.allclose(LSE[live], LSEb[live], rtol=1e-12, atol=1e-13)
    assert np.all(O[~live] == 0)


def test_naive_softmax_matches_safe_tiny():
    rng = np.random.default_rng(7)
    for _ in range(20):
        s = rng.normal(scale=30.0, size=rng.integers(1, 64))
        assert np.allclose(oracle.softmax_naive(s), oracle.softmax_safe(s), rtol=1e-12, atol=1e-300)


def test_lse_against_scipy_logsumexp():
    rng = np.random.default_rng(11)
    Q, K, V = rng.normal(size=(6, 8)), rng.normal(size=(10, 8)), rng.normal(size=(10, 8))
    scale = 0.3
    _, LSE = oracle.attention_head(Q, K, V, scale, causal=True)
    S = scale * Q @ K.T
    for i in range(6):
        vis = oracle.visible_row(i, 6, 10, True)
        assert abs(LSE[i] - logsumexp(S[i][vis])) < 1e-12


def test_attention_rows_matches_attention():
    rng = np.random.default_rng(3)
    B, H, Nq, Nk, d = 2, 2, 9, 11, 4
    Q, K, V = (rng.normal(size=(B, H, n, d)) for n in (Nq, Nk, Nk))
    lens = np.array([0, 7])
    O, LSE = oracle.attention(Q, K, V, 0.5, True, lens)
    picks = [(b, h, i) for b in range(B) for h in range(H) for i in range(Nq)]
    Or, LSEr = oracle.attention_rows(Q, K, V, 0.5, True, lens, picks)
    assert np.allclose(Or, O.reshape(-1, d), rtol=1e-12, atol=1e-14)
    assert np.array_equal(np.isinf(LSEr), np.isinf(LSE.reshape(-1)))
    fin = np.isfinite(LSEr)
    assert np.allclose(LSEr[fin], LSE.reshape(-1)[fin], rtol=1e-12)


def test_attention_rows_any_order_and_chunking_against_brute_force():
    """Rows picked out of order, repeated, over several heads and cut into chunks of three
    must each equal the brute-force definition, in the order they were asked for."""
    rng = np.random.default_rng(5)
    B, H, Nq, Nk, d = 2, 3, 10, 13, 4
    Q, K, V = (rng.normal(size=(B, H, n, d)) for n in (Nq, Nk, Nk))
    lens = np.array([9, 0])
    picks = [(1, 2, 3), (0, 1, 9), (0, 1, 0), (0, 0, 5), (0, 1, 9), (1, 0, 9), (0, 2, 4), (0, 1, 7), (0, 1, 2)]
    for causal in (False, True):
        Or, LSEr = oracle.attention_rows(Q, K, V, 0.5, causal, lens, picks, chunk=3)
        for r, (b, h, i) in enumerate(picks):
            Ob, LSEb = brute_force(Q[b, h], K[b, h], V[b, h], 0.5, causal, int(lens[b]))
            assert np.allclose(Or[r], Ob[i], rtol=1e-12, atol=1e-14), (causal, r)
            if np.isfinite(LSEb[i]):
                assert abs(LSEr[r] - LSEb[i]) < 1e-12
            else:
                assert np.isneginf(LSEr[r]) and np.all(Or[r] == 0)


def test_visible_rows_are_rows_of_visible():
    for causal, L in ((False, None), (True, None), (True, 5), (False, 0)):
        full = np.broadcast_to(oracle.visible(7, 9, causal, L), (7, 9))  # [1, Nk] without a causal mask
        rows = [6, 0, 3, 3]
        assert np.array_equal(oracle.visible_rows(rows, 7, 9, causal, L), full[rows])


def test_bf16_decode():
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x7F80 = +inf, 0x0001 = smallest subnormal 2^-133
    got = oracle.bf16_to_f64(np.array([0x3F80, 0xC000, 0x7F80, 0x0001, 0x4049], dtype=np.uint16))
    assert got[0] == 1.0 and got[1] == -2.0 and np.isinf(got[2]) and got[3] == 2.0 ** -133
    assert got[4] == 3.140625
    import torch
    codes = np.arange(0, 65536, 97, dtype=np.uint16)
    ref = torch.from_numpy(codes.astype(np.int32).astype(np.int16)).view(torch.bfloat16).double().numpy()
    mine = oracle.bf16_to_f64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(mine[fin], ref[fin])


# ---------------------------------------------------------------- invariants

def test_shift_invariance():
    rng = np.random.default_rng(5)
    s = rng.normal(size=37)
    for c in (-800.0, -3.0, 0.5, 650.0):
        assert np.allclose(oracle.softmax_safe(s + c), oracle.softmax_safe(s), rtol=1e-12)


@pytest.mark.parametrize("block", [1, 2, 3, 5, 8, 64])
def test_block_size_and_order_invariance(block):
    rng = np.random.default_rng(block)
    N, dv = 50, 3
    s = rng.normal(scale=4.0, size=N)
    v = rng.normal(size=(N, dv))
    ref = softmax_weights_times(s, v)
    o, _, _ = oracle.online_softmax_attention(s, v, block)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-14)
    nblk = (N + block - 1) // block
    for order in (list(range(nblk))[::-1], list(rng.permutation(nblk))):
        o2, _, _ = oracle.online_softmax_attention(s, v, block, order=order)
        assert np.allclose(o2, ref, rtol=1e-12, atol=1e-14)


def softmax_weights_times(s, v):
    return oracle.softmax_safe(s) @ v


def test_max_in_first_vs_last_tile():
    # moderate scores, then the largest one placed first and then last
    base = np.full(64, 1.0)
    base[::7] = -2.0
    v = np.arange(64, dtype=float)[:, None] * 0.1
    first = base.copy(); first[0] = 30.0
    last = base.copy(); last[-1] = 30.0
    for s in (first, last):
        for block in (4, 16, 64):
            o, _, _ = oracle.online_softmax_attention(s, v, block)
            assert np.allclose(o, oracle.softmax_safe(s) @ v, rtol=1e-12)


def test_state_bounds_alpha_p_in_unit_interval():
    rng = np.random.default_rng(9)
    s = rng.normal(scale=50.0, size=200)
    tr = []
    oracle.online_softmax_attention(s, rng.normal(size=200), 16, trace=tr)
    for t in tr:
        assert 0.0 <= t["alpha"] <= 1.0
        assert np.all((t["p"] >= 0.0) & (t["p"] <= 1.0))
    # loop invariant: after each block, (m, l) equal the stats of the prefix
    for t in tr:
        m, l = oracle.softmax_stats(s[:16 * (t["block"] + 1)])
        assert t["m"] == m and abs(t["l"] - l) <= 1e-12 * l


def test_closed_forms():
    rng = np.random.default_rng(13)
    Q, K = rng.normal(size=(7, 5)), rng.normal(size=(9, 5))
    # V = 1: every live row sums to one
    O, _ = oracle.attention_head(Q, K, np.ones((9, 5)), 0.4, causal=True)
    assert np.allclose(O, 1.0, rtol=1e-13)
    # identical keys: uniform weights, output is the mean of V over visible keys
    Kc = np.tile(K[:1], (9, 1))
    V = rng.normal(size=(9, 5))
    O, LSE = oracle.attention_head(Q, Kc, V, 0.4)
    assert np.allclose(O, V.mean(axis=0), rtol=1e-12)
    assert np.allclose(LSE, 0.4 * Q @ K[0] + math.log(9), rtol=1e-12)
    # one visible key: output is that key's value, LSE its score
    O, LSE = oracle.attention_head(Q, K, V, 0.4, key_len=1)
    assert np.allclose(O, V[0]) and np.allclose(LSE, 0.4 * Q @ K[0])


def test_masks_padding_equals_truncation_and_full_mask():
    rng = np.random.default_rng(17)
    Q, K, V = rng.normal(size=(6, 4)), rng.normal(size=(10, 4)), rng.normal(size=(10, 4))
    for L in (1, 4, 9, 10):
        O, LSE = oracle.attention_head(Q, K, V, 0.5, key_len=L)
        Ot, LSEt = oracle.attention_head(Q, K[:L], V[:L], 0.5)
        assert np.allclose(O, Ot, rtol=1e-13) and np.allclose(LSE, LSEt, rtol=1e-13)
    for L in (0, -3):
        O, LSE = oracle.attention_head(Q, K, V, 0.5, key_len=L)
        assert np.all(O == 0.0) and np.all(LSE == -np.inf)
    O, LSE = oracle.attention_head(Q, K[:0], V[:0], 0.5)
    assert O.shape == (6, 4) and np.all(O == 0.0) and np.all(LSE == -np.inf)
    # causal, Nq = Nk: row i is the unmasked attention over the prefix 0..i
    Qs = rng.normal(size=(10, 4))
    O, LSE = oracle.attention_head(Qs, K, V, 0.5, causal=True)
    for i in range(10):
        Oi, Li = oracle.attention_head(Qs[i:i + 1], K[:i + 1], V[:i + 1], 0.5)
        assert np.allclose(O[i], Oi[0], rtol=1e-13) and abs(LSE[i] - Li[0]) < 1e-13


def test_masked_key_leakage():
    # a masked key with a huge score and a huge value must change nothing
    rng = np.random.default_rng(19)
    s = rng.normal(size=20)
    v = rng.normal(size=(20, 2))
    s2, v2 = s.copy(), v.copy()
    s2[13], v2[13] = 1000.0, 1e4
    valid = np.ones(20, bool); valid[13] = False
    ref, _, _ = oracle.online_softmax_attention(np.delete(s, 13), np.delete(v, 13, 0), 4)
    for block in (4, 7, 20):
        o, _, _ = oracle.online_softmax_attention(s2, v2, block, valid=valid)
        assert np.allclose(o, ref, rtol=1e-12)


def test_huge_scores_stay_finite():
    rng = np.random.default_rng(23)
    Q = rng.normal(size=(4, 8)) * 40
    K = rng.normal(size=(16, 8)) * 40
    V = rng.normal(size=(16, 8))
    O, LSE = oracle.attention_head(Q, K, V, 1.0 / math.sqrt(8))
    S = Q @ K.T / math.sqrt(8)
    assert S.max() > 710  # naive exp would be inf here
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(LSE))
    for i in range(4):
        assert np.allclose(O[i], oracle.softmax_safe(S[i]) @ V, rtol=1e-12)


# ---------------------------------------------------------------- planted mistakes

def _catches(run) -> bool:
    try:
        run()
    except AssertionError:
        return True
    return False


def test_mutation_rescale_l_only_is_caught(golden):
    g = golden["attention_rescale"]
    def run():
        o, _, _ = oracle.online_softmax_attention(g["scores"], np.array(g["V"], float), 2, _mutation="rescale_l_only")
        assert np.allclose(o, g["output_verification"], atol=1e-3)
    assert _catches(run)


def test_mutation_local_max_is_caught(golden):
    g = golden["blocks_2413"]
    _, _, l = oracle.online_softmax_attention(sum(g["blocks"], []), np.zeros(4), 2, _mutation="local_max")
    assert abs(l - g["naive_wrong_sum_reading"]) <= g["tol"]   # reproduces the page's wrong total
    assert abs(l - g["after"][-1]["l"]) > 0.5


def test_mutation_normalize_per_block_is_caught(golden):
    g = golden["scalar_values"]
    o, _, _ = oracle.online_softmax_attention(g["scores"], g["v"], 2, _mutation="normalize_per_block")
    assert abs(o - g["o"]) > 10 * g["tol_o"]   # 36.59 against the printed 36.88


def test_mutation_finite_init_is_caught():
    # all scores far below a finite initial max: every p underflows and the
    # row comes back empty, which the shift-invariance pin rejects
    s = np.array([-2.0, 0.0, -3.0, -1.0]) - 800.0
    v = np.array([1.0, 2.0, 3.0, 4.0])
    good, _, _ = oracle.online_softmax_attention(s, v, 2)
    bad, _, _ = oracle.online_softmax_attention(s, v, 2, _mutation="finite_init")
    want = oracle.softmax_safe(s + 800.0) @ v
    assert abs(good - want) < 1e-12
    assert abs(bad - want) > 1.0


def test_mutation_mask_after_max_is_caught():
    rng = np.random.default_rng(29)
    s = rng.normal(size=12)
    v = rng.normal(size=12)
    s[5] = 1000.0
    valid = np.ones(12, bool); valid[5] = False
    want = oracle.softmax_safe(np.delete(s, 5)) @ np.delete(v, 5)
    good, _, _ = oracle.online_softmax_attention(s, v, 4, valid=valid)
    bad, _, _ = oracle.online_softmax_attention(s, v, 4, valid=valid, _mutation="mask_after_max")
    assert abs(good - want) < 1e-12
    assert not abs(bad - want) < 1e-6


def _threshold_recurrence(s, v, block, tau):
    """The block-wise update with a reference that moves only when a block max passes it
    by more than tau (the library's lazy-rescale option); returns the largest p, l and
    |o~| met on the way and the final (o, l)."""
    m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
    pmax = lmax = omax = 0.0
    for lo in range(0, len(s), block):
        sb, vb = s[lo:lo + block], v[lo:lo + block]
        mb = sb.max()
        m_new = mb if mb > m + tau else m
        alpha = np.exp(m - m_new) if m > -np.inf else 0.0
        p = np.exp(sb - m_new)
        l = alpha * l + p.sum()
        o = alpha * o + p @ vb
        m = m_new
        pmax, lmax, omax = max(pmax, p.max()), max(lmax, l), max(omax, np.abs(o).max())
    return pmax, lmax, omax, o / l, l


@pytest.mark.parametrize("tau", [0.0, 5.5, 20.0])
def test_lazy_rescale_stability_bound(tau):
    """The bound stated for the lazy-rescale option ("FlashAttention math", "Proof of
    numerical stability", restated for a reference that trails the max by up to tau):
    p <= e^tau, l <= Nk e^tau, |o~| <= Nk e^tau max|V|; and the result is the softmax."""
    rng = np.random.default_rng(int(tau * 10) + 1)
    Nk, block = 1024, 128
    v = rng.uniform(-100.0, 100.0, size=(Nk, 8))
    cases = [rng.normal(scale=3.0, size=Nk),
             (tau - 1e-9) * (np.arange(Nk) // block) + 0.0,          # rises by just under tau per block
             (tau + 0.5) * (np.arange(Nk) // block) + rng.normal(scale=0.1, size=Nk)]
    bound = math.exp(tau)
    for s in cases:
        pmax, lmax, omax, out, _ = _threshold_recurrence(s, v, block, tau)
        assert pmax <= bound * (1 + 1e-12)
        assert lmax <= Nk * bound * (1 + 1e-12)
        assert omax <= Nk * bound * np.abs(v).max() * (1 + 1e-12)
        O, _ = oracle.attention_head(np.array([[1.0]]), s[:, None], v, 1.0)
        assert np.allclose(out, O[0], rtol=1e-10, atol=1e-9)
    # the case that rises by just under tau reaches the bound within a factor e^-1e-9
    pmax, *_ = _threshold_recurrence(cases[1], v, block, tau)
    assert pmax >= bound * math.exp(-1e-6)
