"""Pins of the oracle's partial states and their merge (the split-KV path).

A state (m, l, o~) summarises the keys of one range ("FlashAttention math",
section "The running state"); merging states of disjoint ranges uses the rescaling
identity of the same page.  The pins: the pages' printed per-block states and the
final values of their two worked examples, merged in either order; the three-pass
oracle for random partitions (the pages' "Proof of exactness": block size and order
do not change the result); closed forms for one visible key and for empty ranges;
and planted mistakes that a pin must catch.
"""
import itertools

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def one_dim(scores, V):
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(V, dtype=np.float64)
    if v.ndim == 1:
        v = v[:, None]
    return np.ones((1, 1)), s[:, None], v


def block_states(scores, V, block):
    q, k, v = one_dim(scores, V)
    n = len(scores)
    return [oracle.attention_state_head(q, k, v, 1.0, False, None, lo, min(lo + block, n))
            for lo in range(0, n, block)]


def test_scalar_example_block_states_and_merge(golden):
    g = golden["scalar_values"]
    states = block_states(g["scores"], g["v"], g["block"])
    # the first block's state is the state the page prints after block 1
    o1, m1, l1 = states[0]
    assert m1[0] == g["blocks"][0]["m"]
    assert abs(l1[0] - g["blocks"][0]["l"]) <= g["tol"]
    assert abs(o1[0, 0] - g["blocks"][0]["o"]) <= 5e-4
    for order in (states, states[::-1]):
        o, m, l = oracle.merge_states(order)
        assert m[0] == g["blocks"][1]["m"]
        assert abs(l[0] - g["l"]) <= g["tol"]
        assert abs(o[0, 0] - g["o_tilde"]) <= 5e-4
        O, LSE = oracle.finish_state(o, m, l)
        assert abs(O[0, 0] - g["o"]) <= g["tol_o"]


def test_two_dim_rescale_example_merge(golden):
    g = golden["attention_rescale"]
    states = block_states(g["scores"], g["V"], g["block"])
    o1, m1, l1 = states[0]
    a = g["after"][0]
    assert m1[0] == a["m"] and abs(l1[0] - a["l"]) <= g["tol"]
    assert np.allclose(o1[0], a["o"], atol=g["tol"])
    for order in (states, states[::-1]):
        o, m, l = oracle.merge_states(order)
        b = g["after"][1]
        assert m[0] == b["m"] and abs(l[0] - b["l"]) <= g["tol"]
        assert np.allclose(o[0], b["o"], atol=g["tol"])
        O, _ = oracle.finish_state(o, m, l)
        assert np.allclose(O[0], g["output"], atol=2 * g["tol"])


@pytest.mark.parametrize("causal,key_len", [(False, None), (True, None), (False, 37), (True, 50)])
def test_random_partitions_merge_to_three_pass(causal, key_len):
    rng = np.random.default_rng(7)
    Nq, Nk, d = 9, 61, 8
    q = rng.normal(size=(Nq, d))
    k = rng.normal(size=(Nk, d)) * 2.0
    v = rng.normal(size=(Nk, 5))
    O_ref, LSE_ref = oracle.attention_head(q, k, v, 0.7, causal, key_len)
    for trial in range(6):
        cuts = sorted(rng.integers(0, Nk + 1, size=trial + 1).tolist())
        bounds = [0] + cuts + [Nk]
        states = [oracle.attention_state_head(q, k, v, 0.7, causal, key_len, lo, hi)
                  for lo, hi in zip(bounds[:-1], bounds[1:])]
        rng.shuffle(states)
        O, LSE = oracle.finish_state(*oracle.merge_states(states))
        assert np.allclose(O, O_ref, rtol=1e-12, atol=1e-13)
        live = np.isfinite(LSE_ref)
        assert np.array_equal(np.isfinite(LSE), live)
        assert np.allclose(LSE[live], LSE_ref[live], rtol=0, atol=1e-12)


def test_merge_is_order_free_and_associative():
    rng = np.random.default_rng(8)
    q, k, v = rng.normal(size=(4, 6)), rng.normal(size=(40, 6)) * 3, rng.normal(size=(40, 3))
    parts = [oracle.attention_state_head(q, k, v, 1.0, False, None, lo, lo + 10) for lo in range(0, 40, 10)]
    ref = oracle.finish_state(*oracle.merge_states(parts))
    for perm in itertools.permutations(range(4)):
        got = oracle.finish_state(*oracle.merge_states([parts[i] for i in perm]))
        assert np.allclose(got[0], ref[0], rtol=1e-13, atol=1e-14)
    nested = oracle.merge_states([oracle.merge_states(parts[:2]), oracle.merge_states(parts[2:])])
    assert np.allclose(oracle.finish_state(*nested)[0], ref[0], rtol=1e-13, atol=1e-14)


def test_closed_forms_one_key_and_empty_ranges():
    q, k, v = one_dim([3.5, -1.0], [[2.0, -4.0], [1.0, 1.0]])
    o, m, l = oracle.attention_state_head(q, k, v, 1.0, False, None, 0, 1)
    assert m[0] == 3.5 and l[0] == 1.0 and np.array_equal(o[0], [2.0, -4.0])
    empty = oracle.attention_state_head(q, k, v, 1.0, False, None, 1, 1)
    assert empty[1][0] == -np.inf and empty[2][0] == 0.0 and not empty[0].any()
    # padding hides key 1: the range [1, 2) is empty although it holds a key
    hidden = oracle.attention_state_head(q, k, v, 1.0, False, 1, 1, 2)
    assert hidden[1][0] == -np.inf and hidden[2][0] == 0.0
    merged = oracle.merge_states([(o, m, l), empty, hidden])
    assert merged[1][0] == 3.5 and merged[2][0] == 1.0 and np.array_equal(merged[0][0], [2.0, -4.0])
    O, LSE = oracle.finish_state(*oracle.merge_states([empty, hidden]))
    assert not O.any() and LSE[0] == -np.inf


def test_batched_states_match_per_head():
    rng = np.random.default_rng(9)
    Q = rng.normal(size=(2, 2, 5, 4))
    K = rng.normal(size=(2, 2, 7, 4))
    V = rng.normal(size=(2, 2, 7, 3))
    ranges = [(0, 3), (3, 7)]
    o, m, l = oracle.attention_states(Q, K, V, 0.5, True, [7, 4], ranges)
    O_ref, LSE_ref = oracle.attention(Q, K, V, 0.5, True, [7, 4])
    O, LSE = oracle.finish_state(*oracle.merge_states([(o[s], m[s], l[s]) for s in range(2)]))
    assert np.allclose(O, O_ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(LSE, LSE_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mutation", ["rescale_l_only", "no_rescale"])
def test_merge_mutations_are_caught(golden, mutation):
    g = golden["scalar_values"]
    states = block_states(g["scores"], g["v"], g["block"])
    o, m, l = oracle.merge_states(states, _mutation=mutation)
    O, _ = oracle.finish_state(o, m, l)
    assert abs(O[0, 0] - g["o"]) > 10 * g["tol_o"]
