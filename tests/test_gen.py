"""The seeded input generator: its stream, its distributions, bf16 rounding, the workloads."""
import numpy as np
import pytest
import torch

import gen


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 seeded with 1234567 (the reference sequence
    # printed with Vigna's splitmix64.c / Java's SplittableRandom mixer)
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [int(x) for x in gen.splitmix64_sequence(5, 1234567)] == want


def test_streams_are_deterministic_and_distinct():
    a = gen.raw_u64(1000, 42, 0)
    assert np.array_equal(a, gen.raw_u64(1000, 42, 0))
    assert not np.array_equal(a, gen.raw_u64(1000, 42, 1))
    assert not np.array_equal(a, gen.raw_u64(1000, 43, 0))
    # counter-based: a prefix is the same whatever the length drawn
    assert np.array_equal(gen.raw_u64(10, 42, 0), a[:10])
    # multithreaded fill equals the single-threaded prefix
    big = gen.normal_bf16((1 << 17,), 5, 2)
    assert np.array_equal(big[:1000], gen.normal_bf16((1000,), 5, 2))


def test_normal_moments():
    x = gen.codes_to_f32(gen.normal_bf16((1 << 18,), 1, 0, 0.0, 1.0)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    y = gen.codes_to_f32(gen.normal_bf16((1 << 18,), 1, 0, 0.0, 0.5)).astype(np.float64)
    assert abs(y.std() - 0.5) < 0.005
    # fourth moment of a normal is 3 sigma^4
    assert abs((x ** 4).mean() - 3.0) < 0.1


def test_uniform_range_and_ints():
    u = gen.codes_to_f32(gen.uniform_bf16((1 << 16,), 3, 2, -100.0, 100.0))
    assert u.min() >= -100.0 and u.max() <= 100.0 and abs(u.mean()) < 1.5
    ints = gen.uniform_int(20000, 9, 3, 1, 4095)
    assert ints.min() >= 1 and ints.max() <= 4095
    assert abs(ints.mean() - 2048) < 40


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=5000).astype(np.float32),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0, 65504.0], np.float32)])
    mine = gen.f32_to_codes(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(mine, ref)
    # ties go to even: 1 + 2^-8 -> 1.0 (0x3F80); 1 + 3*2^-8 -> 0x3F82
    assert mine[-4] == 0x3F80 and mine[-3] == 0x3F82


@pytest.mark.parametrize("name", ["b1h2n256d64", "padded_planted_b2h8n4096d128"])
def test_workloads_shapes_and_determinism(name):
    a = gen.make_inputs(name)
    b = gen.make_inputs(name)
    w = gen.WORKLOADS[name]
    assert a["Q"].shape == (w["B"], w["H"], w["Nq"], w["d"]) and a["Q"].dtype == np.uint16
    for t in ("Q", "K", "V"):
        assert np.array_equal(a[t], b[t])


def test_planted_workload_structure():
    x = gen.make_inputs("padded_planted_b2h8n4096d128")
    lens = x["lens"]
    assert lens[0] == 0 and 1 <= lens[1] <= 4095
    V = gen.codes_to_f32(x["V"])
    assert V.min() >= -100 and V.max() <= 100
    jstar = x["planted_key"]
    assert np.all(jstar[0] == -1)
    L = int(lens[1])
    rows = np.arange(x["Nq"])
    j1 = jstar[1]
    assert np.all(j1[:, rows % 2 == 0] < min(128, L))
    assert np.all(j1[:, rows % 2 == 1] >= max(0, L - 128)) and np.all(j1 < L)
    # the planted score is close to 60 and is the row maximum over valid keys
    for h in (0, 5):
        q = gen.codes_to_f32(x["Q"][1, h]).astype(np.float64)
        k = gen.codes_to_f32(x["K"][1, h, :L]).astype(np.float64)
        s = x["scale"] * q @ k.T
        planted = s[rows, j1[h]]
        assert np.all(np.abs(planted - 60.0) < 1.0)
        assert np.all(np.argmax(s, axis=1) == j1[h])
