"""The d = 64 forward with two query tiles per CTA, against the fp64 oracle.

At d = 64 the library runs two adjacent query tiles per CTA once the pairs of tiles are
at least as many as the SMs (causal) or more than half of them (no causal mask); smaller
problems keep one tile per CTA.  Every case here is above that threshold, so it runs the
two-tile kernel, with odd tile counts (a pair whose
second tile lies past the end), tail rows, padded and fully masked batches, bottom-right
causal masks with Nq > Nk (a pair whose first tile sees no key while the second does)
and Nq < Nk, packed sequences, a strided layout, the options of attn_fwd_ex and the
timeout path.  The per-row arithmetic is the one-tile kernel's, so the two must agree bit
for bit: the last tests run a problem once whole (two tiles per CTA) and once a batch at
a time (too few pairs, one tile per CTA) and compare the bytes.
"""
import ctypes
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, run_cuda, to_device

pytestmark = pytest.mark.gpu


def custom(B, H, Nq, Nk, causal=False, seed=7, lens=None):
    w = dict(name="custom", B=B, H=H, Nq=Nq, Nk=Nk, d=64, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None if lens is None else ("given", lens), plant=None,
             scale=1.0 / math.sqrt(64))
    return gen.make_inputs(w)


def sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def pairs(B, H, Nq):
    return B * H * ((-(-Nq // 128) + 1) // 2)


def takes_pair_kernel(B, H, Nq, causal):
    """The library's rule: causal, at least one pair per SM; otherwise more than half."""
    n = pairs(B, H, Nq)
    return n >= sms() if causal else 2 * n > sms()


CASES = [
    # B, H, Nq, Nk, causal, lens
    (4, 40, 300, 300, True, None),                 # 3 tiles per head: the second pair has one tile
    (4, 40, 512, 700, False, [700, 0, 129, 1]),    # padding, one fully masked batch, Nk tail
    (2, 80, 384, 256, True, None),                 # Nq > Nk: the first tile of each head sees no key
    (2, 80, 256, 640, True, None),                 # Nq < Nk
    (1, 160, 200, 200, False, [150]),              # one pair per head, the second tile short
    (2, 48, 1024, 1024, True, None),               # several blocks per tile, several pairs per CTA
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal,lens", CASES)
def test_two_tile_kernel_matches_oracle(B, H, Nq, Nk, causal, lens):
    assert takes_pair_kernel(B, H, Nq, causal), "the case must take the two-tile kernel"
    x = custom(B, H, Nq, Nk, causal, seed=1300 + B * H + Nq + Nk, lens=lens)
    O, LSE = run_cuda(x)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O, LSE, O_ref, LSE_ref)


def _one_batch_at_a_time(x, causal, lens):
    """The same problem one batch per call: B * H pairs drop below the SM count."""
    outs, lses = [], []
    for b in range(x["Q"].shape[0]):
        xb = dict(x, Q=x["Q"][b:b + 1], K=x["K"][b:b + 1], V=x["V"][b:b + 1])
        O, LSE = run_cuda(xb, causal=causal, lens=None if lens is None else [lens[b]])
        outs.append(O)
        lses.append(LSE)
    return np.concatenate(outs), np.concatenate(lses)


@pytest.mark.parametrize("B,H,Nq,Nk,causal,lens", [
    (4, 40, 300, 300, True, None),
    (4, 36, 512, 700, False, [700, 0, 129, 1]),
    (2, 72, 384, 256, True, None),
])
def test_two_tile_kernel_equals_one_tile_kernel_bitwise(B, H, Nq, Nk, causal, lens):
    x = custom(B, H, Nq, Nk, causal, seed=1400 + Nq, lens=lens)
    assert takes_pair_kernel(B, H, Nq, causal) and not takes_pair_kernel(1, H, Nq, causal)
    O2, L2 = run_cuda(x)
    O1, L1 = _one_batch_at_a_time(x, causal, lens)
    assert np.array_equal(O1, O2)
    assert np.array_equal(L1, L2)


def test_two_tile_kernel_packed_sequences():
    """Packed sequences at d = 64: 90 of them, 4 heads, lengths 0..700 (pairs past the end
    of the shorter sequences are skipped)."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    rng = np.random.default_rng(15)
    H, d, n = 4, 64, 90
    lq = rng.integers(0, 700, size=n)
    lk = lq + rng.integers(0, 100, size=n)
    assert takes_pair_kernel(n, H, int(lq.max()), True)
    total_q, total_k = int(lq.sum()), int(lk.sum())
    w = dict(name="packed", B=1, H=H, Nq=total_q, Nk=total_k, d=d, causal=False, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=33, lens=None, plant=None, scale=1.0 / math.sqrt(d))
    x = gen.make_inputs(w)
    Qp = np.ascontiguousarray(x["Q"][0].transpose(1, 0, 2))   # [total_q, H, d]
    Kp = np.ascontiguousarray(x["K"][0].transpose(1, 0, 2))
    Vp = np.ascontiguousarray(x["V"][0].transpose(1, 0, 2))
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    O, LSE = pkg.attn_fwd_varlen(to_device(Qp), to_device(Kp), to_device(Vp), torch.from_numpy(cu_q).cuda(),
                                 torch.from_numpy(cu_k).cuda(), int(lq.max()), scale=x["scale"], causal=True)
    pkg.status_sync()
    Of = O.float().cpu().numpy().astype(np.float64)
    Lf = LSE.cpu().numpy().astype(np.float64)
    for b in range(n):
        if lq[b] == 0:
            continue
        rq, rk = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        O_ref = np.zeros((H, lq[b], d))
        L_ref = np.zeros((H, lq[b]))
        for h in range(H):
            O_ref[h], L_ref[h] = oracle.attention_head(oracle.bf16_to_f64(Qp[rq, h]), oracle.bf16_to_f64(Kp[rk, h]),
                                                       oracle.bf16_to_f64(Vp[rk, h]), x["scale"], True)
        compare(Of[rq].transpose(1, 0, 2), Lf[:, rq], O_ref, L_ref)


def test_two_tile_kernel_bshd_layout():
    """[B, N, H, d] through attn_fwd_strided equals the contiguous call bit for bit."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    B, H, N = 2, 80, 384
    x = custom(B, H, N, N, True, seed=1500)
    O_ref, L_ref = run_cuda(x)
    Q, K, V = (to_device(x[k]).transpose(1, 2).contiguous() for k in ("Q", "K", "V"))   # [B, N, H, d]
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((B, H, N), float("nan"), device="cuda")
    pkg.attn_fwd_strided(Q.transpose(1, 2), K.transpose(1, 2), V.transpose(1, 2), O.transpose(1, 2), LSE,
                         scale=x["scale"], causal=True)
    pkg.status_sync()
    assert np.array_equal(O.transpose(1, 2).float().cpu().numpy().astype(np.float64), O_ref)
    assert np.array_equal(LSE.cpu().numpy().astype(np.float64), L_ref)


@pytest.mark.parametrize("tau,mode", [(4.0, 0), (0.0, 2), (4.0, 2)])
def test_two_tile_kernel_options(tau, mode):
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    B, H, N = 2, 80, 512
    x = custom(B, H, N, N + 100, True, seed=1600 + mode, lens=[N + 100, 333])
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, N), device="cuda")
    lt = torch.tensor(x["lens"], dtype=torch.int32, device="cuda")
    pkg.attn_fwd(Q, K, V, O, LSE, scale=x["scale"], causal=True, key_padding_lens=lt,
                 rescale_threshold=tau, exp2_mode=mode)
    pkg.status_sync()
    O_ref, L_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], True, x["lens"])
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, L_ref)


def test_two_tile_kernel_withheld_block_times_out(monkeypatch):
    """The timeout path of the two-tile kernel: a withheld K block ends every wait on it,
    the status word reports ATTN_ERR_TIMEOUT, and the next call is correct."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    B, H, N = 2, 80, 256
    x = custom(B, H, N, N, False, seed=1700)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, N), device="cuda")
    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "100")
    monkeypatch.setenv("ATTN_ENABLE_TEST_HOOKS", "1")
    monkeypatch.setenv("ATTN_TEST_WITHHOLD_K_BLOCK", "1")
    pkg.attn_fwd(Q, K, V, O, LSE, scale=x["scale"])
    with pytest.raises(pkg.AttnError) as err:
        pkg.status_sync()
    assert err.value.status == -7
    pkg.status_sync()
    monkeypatch.delenv("ATTN_TEST_WITHHOLD_K_BLOCK")
    monkeypatch.delenv("ATTN_WAIT_LIMIT_MS")
    O2, L2 = run_cuda(x)
    O_ref, L_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], False, None)
    compare(O2, L2, O_ref, L_ref)


def test_two_tile_kernel_random_shapes_bitwise():
    """Seeded random shapes (tile counts 1..9, ragged Nq, Nk from 0, causal or not, padding
    lengths from 0 to past Nk): the two-tile kernel on the whole problem equals the one-tile
    kernel run a batch at a time, bit for bit."""
    rng = np.random.default_rng(2024)
    n_sm = sms()
    for case in range(14):
        nqt = int(rng.integers(1, 10))
        per_head = (nqt + 1) // 2
        causal = bool(rng.integers(0, 2))
        # one batch stays below the two-tile threshold, the whole problem reaches the SM count
        H = max(1, ((n_sm - 1) if causal else (n_sm // 2)) // per_head)
        B = -(-n_sm // (H * per_head)) + int(rng.integers(0, 3))
        Nq = int(rng.integers(max(1, 128 * (nqt - 1) + 1), 128 * nqt + 1))
        Nk = int(rng.integers(0, 1500))
        lens = None
        if rng.integers(0, 2):
            lens = [int(v) for v in rng.integers(0, Nk + 200, size=B)]
            lens[int(rng.integers(0, B))] = 0
        assert takes_pair_kernel(B, H, Nq, causal) and not takes_pair_kernel(1, H, Nq, causal)
        x = custom(B, H, Nq, Nk, causal, seed=1800 + case, lens=lens)
        O2, L2 = run_cuda(x)
        O1, L1 = _one_batch_at_a_time(x, causal, lens)
        assert np.array_equal(O1, O2), (case, B, H, Nq, Nk, causal, lens)
        assert np.array_equal(L1, L2), (case, B, H, Nq, Nk, causal, lens)
