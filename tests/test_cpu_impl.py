"""The CPU library (libattn_cpu.so, include/attn_cpu.h) against the fp64 oracle, on the
host: the blocked online-softmax recurrence in fp32 with a bf16 output must meet the
same tolerance as the GPU path, on ragged shapes, masks and the fully masked convention.
"""
import math
import os
import re

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    import online_softmax_flashattention_attention_gb300 as p
    from online_softmax_flashattention_attention_gb300 import build as b
    b.build_cpu_library()
    p.load_cpu_library()
    return p


def custom(B, H, Nq, Nk, d, causal=False, seed=7, lens=None, qk=("normal", 0.0, 1.0), v=("normal", 0.0, 1.0)):
    w = dict(name="custom", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=qk, v=v, seed=seed,
             lens=None if lens is None else ("given", lens), plant=None, scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def run(pkg, x, threads=0):
    O, LSE = pkg.attn_fwd_cpu(x["Q"], x["K"], x["V"], scale=x["scale"], causal=x["causal"],
                              key_padding_lens=x["lens"], num_threads=threads)
    return oracle.bf16_to_f64(O), LSE.astype(np.float64)


SHAPES = [
    (1, 2, 256, 256, 64, False, None),
    (2, 3, 130, 130, 128, True, None),
    (1, 2, 200, 65, 128, True, None),         # Nq > Nk: leading rows fully masked
    (1, 1, 63, 300, 128, True, None),         # Nq < Nk
    (3, 1, 100, 200, 64, False, [0, 1, 129]),
    (1, 1, 1, 1, 32, False, None),
    (1, 2, 70, 90, 96, True, None),           # a head size the GPU path does not take
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,lens", SHAPES)
def test_cpu_matches_oracle(pkg, B, H, Nq, Nk, d, causal, lens):
    x = custom(B, H, Nq, Nk, d, causal, seed=Nq + Nk + d, lens=lens)
    O, LSE = run(pkg, x, threads=3)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O, LSE, O_ref, LSE_ref)


def test_cpu_threads_do_not_change_the_result(pkg):
    x = custom(2, 2, 300, 300, 64, True, seed=5)
    a = run(pkg, x, threads=1)
    b = run(pkg, x, threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_cpu_no_keys_and_huge_scores(pkg):
    x = custom(1, 2, 40, 0, 64, False, seed=6)
    O, LSE = run(pkg, x)
    assert not O.any() and np.all(np.isneginf(LSE))
    x = custom(1, 2, 128, 256, 128, False, seed=13, qk=("normal", 0.0, 16.0))   # scores far past 88
    O, LSE = run(pkg, x)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(LSE))
    assert np.abs(O - O_ref).max() <= 2e-2 and np.abs(LSE - LSE_ref).max() <= 1e-3 * np.abs(LSE_ref).max() / 100 + 1e-3


def test_cpu_page_example(pkg, golden):
    # "FlashAttention math", worked example: scores [1, 3, 2, 5], values [10, 20, 30, 40]
    g = golden["scalar_values"]
    d = 8
    q = np.zeros((1, 1, 1, d), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, 4, d), np.float32)
    k[0, 0, :, 0] = g["scores"]
    v = np.zeros((1, 1, 4, d), np.float32)
    v[0, 0, :, 0] = np.array(g["v"], np.float32) / 10.0
    O, LSE = pkg.attn_fwd_cpu(gen.f32_to_codes(q), gen.f32_to_codes(k), gen.f32_to_codes(v), scale=1.0)
    assert abs(float(gen.codes_to_f32(O)[0, 0, 0, 0]) * 10.0 - g["o"]) <= 0.08   # bf16 of 3.688
    assert abs(float(LSE[0, 0, 0]) - (5.0 + math.log(g["l"]))) <= 1e-3


def test_cpu_argument_errors(pkg):
    lib = pkg.load_cpu_library()
    a = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 4, 4, 64, 0.1, 0, None, 1]

    def call(i, v):
        b = list(a)
        b[i] = v
        return lib.attn_fwd_cpu(*b)
    assert call(9, 0) == -3 and call(9, 257) == -3
    assert call(5, -1) == -2
    assert call(10, 0.0) == -8 and call(10, float("nan")) == -8
    assert call(13, -2) == -8
    assert call(0, None) == -1
    assert call(7, 0) == 0          # no query rows: nothing to do


def test_cpu_header_symbols_exported(pkg):
    text = open(os.path.join(ROOT, "include", "attn_cpu.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = sorted(set(re.findall(r"^\s*\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))
    assert names == sorted(pkg.CPU_EXPORTS)
    lib = pkg.load_cpu_library()
    for n in names:
        assert hasattr(lib, n)
