"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on generator
bytes and compare with the fp64 oracle under the tolerance the tests state."""
from __future__ import annotations

import numpy as np

# Tolerance (stated in the workload spec for unit-scale values, widened by half a bf16
# ulp of the reference because O is returned in bf16):
#   |O - O_ref| <= ATOL_O * s_V + ulp_bf16(|O_ref|) / 2   element-wise
#   mean |O - O_ref| <= MEAN_O * s_V
#   |LSE - LSE_ref| <= ATOL_LSE
# s_V is the scale of the values (1 for N(0, sigma <= 1) values, 100 for U[-100, 100]).
ATOL_O = 1e-2
MEAN_O = 1e-3
ATOL_LSE = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 0.5 * np.exp2(e - 7)


def to_device(codes: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(torch.bfloat16).cuda()


def run_cuda(x: dict, causal=None, lens=None, scale=None, fill_nan=True):
    """Run the CUDA forward on the generator's bytes; returns float64 numpy O, LSE."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    B, H, Nq, d = Q.shape
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    if fill_nan:  # unwritten rows show up as NaN
        O.fill_(float("nan"))
        LSE.fill_(float("nan"))
    lens = x.get("lens") if lens is None else lens
    lt = None if lens is None else torch.as_tensor(np.asarray(lens, dtype=np.int32)).cuda()
    pkg.attn_fwd(Q, K, V, O, LSE, scale=x["scale"] if scale is None else scale,
                 causal=x["causal"] if causal is None else causal, key_padding_lens=lt)
    pkg.status_sync()
    return O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64)


def compare(O, LSE, O_ref, LSE_ref, s_v=1.0):
    """Assert the stated tolerance; returns a dict of the observed errors."""
    assert O.shape == O_ref.shape and LSE.shape == LSE_ref.shape
    assert not np.isnan(O).any(), "O has NaN (unwritten or invalid rows)"
    assert not np.isnan(LSE).any(), "LSE has NaN (unwritten or invalid rows)"
    dead = np.isneginf(LSE_ref)
    # fully masked rows: exact convention
    assert np.array_equal(np.isneginf(LSE), dead), "fully-masked rows differ"
    assert np.all(O[dead] == 0.0), "fully-masked rows must have O == 0"
    live = ~dead
    err = np.abs(O - O_ref)
    bound = ATOL_O * s_v + bf16_half_ulp(O_ref)
    worst = float((err / bound).max()) if err.size else 0.0
    assert np.all(err <= bound), f"max |dO| {err.max():.4g} exceeds bound (worst ratio {worst:.3g})"
    mean = float(err.mean()) if err.size else 0.0
    assert mean <= MEAN_O * s_v, f"mean |dO| {mean:.4g} > {MEAN_O * s_v}"
    lerr = np.abs(LSE[live] - LSE_ref[live])
    lmax = float(lerr.max()) if lerr.size else 0.0
    assert lmax <= ATOL_LSE, f"max |dLSE| {lmax:.4g} > {ATOL_LSE}"
    return dict(max_abs_o=float(err.max()) if err.size else 0.0, mean_abs_o=mean, max_abs_lse=lmax,
                worst_ratio=worst)


def sample_rows(B, H, Nq, n_random=24, seed=0):
    """(b, h, i) picks: first/last heads, tile edges, the ends, and random rows."""
    rng = np.random.default_rng(seed)
    rows = sorted({0, 1, 63, 127, 128, 129, Nq // 2, Nq - 129, Nq - 128, Nq - 2, Nq - 1} & set(range(Nq)))
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 2)]
    picks = [(b, h, i) for (b, h) in heads for i in rows]
    for _ in range(n_random):
        picks.append((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(Nq))))
    return sorted(set(picks))
