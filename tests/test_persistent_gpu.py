"""The persistent kernel with several items per CTA, compared whole with the oracle.

The kernel runs one CTA per SM, each walking its items (query tiles, or tiles x key
splits) in a snake order, with the K/V ring, the score buffers and their barrier phases
carried from one item to the next.  The shapes here have two to six times as many
items as the GPU has SMs, mixed with items that have no visible key (fully masked
batches), tail tiles and short sequences, so every CTA crosses several item boundaries.
"""
import math

import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import compare, run_cuda, to_device

pytestmark = pytest.mark.gpu


def custom(B, H, Nq, Nk, d, causal=False, seed=7, lens=None):
    w = dict(name="custom", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=seed, lens=None if lens is None else ("given", lens), plant=None,
             scale=1.0 / math.sqrt(d))
    return gen.make_inputs(w)


def sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


CASES = [
    # B, H, Nq, Nk, d, causal, lens               items = B * H * ceil(Nq / 128)
    (4, 40, 300, 300, 128, True, None),           # 480
    (4, 30, 300, 450, 64, False, [450, 0, 129, 0]),  # 360, half of them with no visible key
    (6, 20, 260, 260, 128, False, [1, 260, 0, 77, 200, 129]),  # 360
    (2, 64, 200, 600, 128, True, None),           # 256, Nq < Nk (bottom-right causal)
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,lens", CASES)
def test_many_items_per_cta(B, H, Nq, Nk, d, causal, lens):
    items = B * H * -(-Nq // 128)
    assert items > sms(), "the case must give CTAs more than one item"
    x = custom(B, H, Nq, Nk, d, causal, seed=900 + B * H + Nq, lens=lens)
    O, LSE = run_cuda(x)
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"])
    compare(O, LSE, O_ref, LSE_ref)


def test_many_items_split_states():
    """Split-KV states with more (tile, split) items than SMs."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    B, H, Nq, Nk, d, S = 2, 40, 256, 900, 128, 3     # 2 * 40 * 2 * 3 = 480 items
    x = custom(B, H, Nq, Nk, d, True, seed=77, lens=[900, 500])
    lt = torch.as_tensor(np.asarray(x["lens"], np.int32)).cuda()
    O, LSE = pkg.attn_fwd_splitkv(to_device(x["Q"]), to_device(x["K"]), to_device(x["V"]), num_splits=S,
                                  scale=x["scale"], causal=True, key_padding_lens=lt)
    pkg.status_sync()
    O_ref, LSE_ref = oracle.attention(x["Q"], x["K"], x["V"], x["scale"], True, x["lens"])
    compare(O.float().cpu().numpy().astype(np.float64), LSE.cpu().numpy().astype(np.float64), O_ref, LSE_ref)


@pytest.mark.parametrize("n,max_len,H,d,seed", [
    (70, 400, 3, 128, 5),    # ranked by work in shared memory (at most 512 sequences)
    (600, 120, 2, 64, 6),    # more than 512: the order of cu_seqlens
])
def test_many_packed_sequences(n, max_len, H, d, seed):
    """Packed sequences of lengths 0..max_len: several items per CTA, many of them past the
    end of their (shorter) sequence; up to 512 sequences the kernel walks them in
    decreasing work, beyond that in the order given."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    rng = np.random.default_rng(seed)
    lq = rng.integers(0, max_len, size=n)
    lk = lq + rng.integers(0, max_len // 2, size=n)
    total_q, total_k = int(lq.sum()), int(lk.sum())
    w = dict(name="packed", B=1, H=H, Nq=total_q, Nk=total_k, d=d, causal=False, qk=("normal", 0.0, 1.0),
             v=("normal", 0.0, 1.0), seed=31, lens=None, plant=None, scale=1.0 / math.sqrt(d))
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


@pytest.mark.parametrize("d", [128, 64])
def test_rank_major_order_leaves_results_unchanged(d):
    """Causal problems whose K and V fit in L2 run every head's longest tiles first (the
    rank-major item order).  A tile's arithmetic does not depend on which CTA runs it or
    when, so the whole problem must equal, bit for bit, its heads run one per call, where
    the order is trivially head major.  (At d = 64 the whole problem takes the two-tile
    kernel and a single head the one-tile kernel; the two agree bit for bit there.)"""
    B, H, N = 2, 40, 700
    lens = [700, 333]
    assert 4 * B * H * N * d <= 96 << 20, "the case must take the rank-major order"
    x = custom(B, H, N, N, d, True, seed=2100 + d, lens=lens)
    O, L = run_cuda(x)
    for b in range(B):
        for h in range(H):
            xs = dict(x, **{k: np.ascontiguousarray(x[k][b:b + 1, h:h + 1]) for k in ("Q", "K", "V")})
            Oh, Lh = run_cuda(xs, lens=[lens[b]])
            assert np.array_equal(Oh[0, 0], O[b, h]), (b, h)
            assert np.array_equal(Lh[0, 0], L[b, h]), (b, h)


@pytest.mark.parametrize("B,H,N,d,causal,lens_kind", [
    (128, 512, 128, 64, False, "mixed"),     # 65536 heads of one tile: bh up to 65535
    (64, 600, 130, 128, True, None),         # 38400 heads of two tiles (the second one row)
])
def test_tens_of_thousands_of_heads_every_item(B, H, N, d, causal, lens_kind):
    """Far more (batch, head) pairs than any other case: the decode's divisions by H and by
    the item-order divisor see numerators up to 76 799.  One row of every work item is
    compared with the oracle (a random row of the tile), plus every row of the last head."""
    lens = None
    if lens_kind == "mixed":
        lens = [int(v) for v in np.random.default_rng(5).integers(0, N + 1, size=B)]
        lens[0], lens[-1] = 0, N
    x = custom(B, H, N, N, d, causal, seed=31 + H, lens=lens)
    O, LSE = run_cuda(x)
    rng = np.random.default_rng(H)
    picks = []
    for b in range(B):
        for h in range(H):
            for t0 in range(0, N, 128):
                picks.append((b, h, int(rng.integers(t0, min(N, t0 + 128)))))
    picks += [(B - 1, H - 1, i) for i in range(N)]
    picks = sorted(set(picks))
    O_ref, LSE_ref = oracle.attention_rows(x["Q"], x["K"], x["V"], x["scale"], causal, x["lens"], picks)
    idx = tuple(np.array(picks).T)
    compare(O[idx], LSE[idx], O_ref, LSE_ref)
    assert np.all(np.isfinite(O))


@pytest.mark.parametrize("B,H,d,causal", [
    (2, 70000, 128, True),      # one-tile kernel: 2.29e9 elements per tensor
    (2, 140000, 64, False),     # two-tile kernel: 2.29e9 elements per tensor
])
def test_tensors_beyond_two_to_the_31_elements(B, H, d, causal):
    """Q, K, V and O each hold more than 2^31 elements (4.6 GB of bf16 each), so the rows of
    the last heads lie past every 32-bit element offset: O's row addresses, the LSE index
    and the tensor maps' head coordinates must all be computed in 64 bits.  Rows of heads
    on both sides of element 2^31 are compared with the oracle; only those rows are copied
    back."""
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    N = 128
    assert B * H * N * d > 2 ** 31
    x = custom(B, H, N, N, d, causal, seed=47 + d)
    Q, K, V = to_device(x["Q"]), to_device(x["K"]), to_device(x["V"])
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    pkg.attn_fwd(Q, K, V, O, LSE, scale=x["scale"], causal=causal)
    pkg.status_sync()
    first_past = (2 ** 31) // (N * d)                 # the first (b, h) whose rows start past 2^31
    bh_picks = sorted({0, H - 1, H, first_past - 1, first_past, first_past + 1, B * H - 2, B * H - 1})
    rng = np.random.default_rng(d)
    bh_picks += [int(v) for v in rng.integers(first_past, B * H, size=6)]
    picks = sorted({(bh // H, bh % H, i) for bh in bh_picks for i in (0, 1, 63, 64, 126, 127)})
    idx = tuple(torch.as_tensor(np.array(picks).T, device="cuda"))
    Os = O[idx].float().cpu().numpy().astype(np.float64)
    Ls = LSE[idx].cpu().numpy().astype(np.float64)
    O_ref, LSE_ref = oracle.attention_rows(x["Q"], x["K"], x["V"], x["scale"], causal, None, picks)
    compare(Os, Ls, O_ref, LSE_ref)
    assert not torch.isnan(O).any().item() and not torch.isnan(LSE).any().item(), "a row was left unwritten"
