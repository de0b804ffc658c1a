"""fp64 CPU oracle of the exact attention forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference`` arm) may import this module.  The
CUDA library never calls it and shares no code with it.

Sources (web pages this module restates):

* [OS] "2.2b: FlashAttention -- Online Softmax" (hf-cn0.pages.dev, blog of
  atharv6f): "The Softmax Formula", "The Numerical Stability Problem",
  "The Sum of Exponentials", "The Key Insight: m and l Are All You Need",
  "The Solution: Rescaling When the Maximum Changes", "Extending to Attention",
  "The Complete Online Softmax Algorithm", "Why This Algorithm is Exact".
* [TA] "Tiled attention: running max softmax" (archcrux.com interview answer):
  masked keys contribute zero; a fully masked row needs a defined convention.
* [FM] "FlashAttention math" (aicassindra.com, transformer_math):
  "What we must compute", "Safe softmax", "The running state",
  "The rescaling identity, derived", "The block-wise update, and the full
  algorithm", "Pitfalls in implementing the recurrence".

Readings where the pages are silent (each is listed in the design notes):

* Scores are s_ij = scale * q_i . k_j with scale = 1/sqrt(d) by default ([FM]
  "What we must compute").  Masked scores are -inf before any maximum is taken
  ([FM] "Pitfalls"), so a masked key is excluded from the max and the sum
  ([TA]).
* Key padding: key j of batch b is visible iff j < L_b (L_b clamped to
  [0, Nk]).  Causal masks are aligned bottom-right: key j is visible to query i
  iff j <= i + (Nk - Nq).
* A fully masked row (no visible key, including Nk = 0) has O = 0 and
  LSE = -inf: the convention [TA] asks for, with values fixed by the workload
  statement.
* LSE = m + ln(l) of the scaled scores; the pages name "logsumexp" but define
  only m and l ([OS] "The Sum of Exponentials").

Every function is pinned by tests in ``tests/test_oracle.py`` and
``tests/test_oracle_states.py`` (partial states and their merge) against the
pages' printed examples, closed forms and brute force.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def bf16_to_f64(codes) -> np.ndarray:
    """Widen raw bf16 codes (uint16) to float64 exactly (bf16 is the top half of an IEEE float32)."""
    u = np.asarray(codes, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# --- softmax of one score vector ---------------------------------------------

def softmax_naive(s) -> np.ndarray:
    """softmax(S)_i = e^{s_i} / sum_j e^{s_j}, no shift ([OS] "The Softmax Formula").

    Overflows to inf/nan once a score passes ~709.78 in float64; that is the
    failure the pages use to motivate the max shift.
    """
    s = np.asarray(s, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(s)
        return e / e.sum()


def softmax_stats(s):
    """(m, l): m = max(S), l = sum_j exp(s_j - m) ([OS] "The Sum of Exponentials").

    For an empty or fully masked vector (max = -inf) returns (-inf, 0.0).
    """
    s = np.asarray(s, dtype=np.float64)
    if s.size == 0:
        return NEG_INF, 0.0
    m = float(np.max(s))
    if m == NEG_INF:
        return NEG_INF, 0.0
    return m, float(np.sum(np.exp(s - m)))


def softmax_safe(s) -> np.ndarray:
    """Three-pass safe softmax: m, then l, then e^{s_i - m} / l ([FM] "Safe softmax")."""
    s = np.asarray(s, dtype=np.float64)
    m, l = softmax_stats(s)
    if l == 0.0:
        return np.zeros_like(s)
    return np.exp(s - m) / l


# --- masks ---------------------------------------------------------------------

def visible(Nq: int, Nk: int, causal: bool, key_len=None) -> np.ndarray:
    """Boolean [Nq, Nk]: may query i attend to key j (padding, then bottom-right causal)."""
    L = Nk if key_len is None else int(min(max(int(key_len), 0), Nk))
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    vis = j < L
    if causal:
        vis = vis & (j <= i + (Nk - Nq))
    return vis


def visible_row(i: int, Nq: int, Nk: int, causal: bool, key_len=None) -> np.ndarray:
    """Row i of ``visible``: boolean [Nk]."""
    L = Nk if key_len is None else int(min(max(int(key_len), 0), Nk))
    j = np.arange(Nk)
    vis = j < L
    if causal:
        vis = vis & (j <= i + (Nk - Nq))
    return vis


# --- attention for one head (the oracle proper) --------------------------------

def attention_head(q, k, v, scale: float, causal: bool = False, key_len=None):
    """Exact attention of one head in float64, three-pass safe softmax per row.

    q [Nq, d], k [Nk, d], v [Nk, dv] (float64).  Returns (O [Nq, dv], LSE [Nq]).

    Pass 1: s = scale * q k^T with masked entries set to -inf, m = row max.
    Pass 2: l = sum_j exp(s_j - m).
    Pass 3: O = sum_j exp(s_j - m) v_j / l;  LSE = m + ln l.
    Rows with no visible key: O = 0, LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Nq, Nk, dv = q.shape[0], k.shape[0], v.shape[1]
    O = np.zeros((Nq, dv), dtype=np.float64)
    LSE = np.full(Nq, NEG_INF, dtype=np.float64)
    if Nq == 0 or Nk == 0:
        return O, LSE
    s = scale * (q @ k.T)
    s = np.where(visible(Nq, Nk, causal, key_len), s, NEG_INF)
    m = s.max(axis=1)                                   # pass 1
    live = m > NEG_INF
    ref = np.where(live, m, 0.0)
    p = np.exp(s - ref[:, None])                        # exp(-inf) = 0 for masked keys
    l = p.sum(axis=1)                                   # pass 2
    acc = p @ v                                         # pass 3
    O[live] = acc[live] / l[live, None]
    LSE[live] = m[live] + np.log(l[live])
    return O, LSE


def attention(Q, K, V, scale: float, causal: bool = False, lens=None):
    """Batched oracle.  Q [B,H,Nq,d], K/V [B,H,Nk,d] as bf16 codes (uint16) or floats.

    Returns float64 O [B,H,Nq,d] and LSE [B,H,Nq].  lens: per-batch key lengths or None.
    """
    Qf, Kf, Vf = (_as_f64(x) for x in (Q, K, V))
    B, H, Nq, _ = Qf.shape
    dv = Vf.shape[3]
    O = np.zeros((B, H, Nq, dv))
    LSE = np.full((B, H, Nq), NEG_INF)
    for b in range(B):
        L = None if lens is None else int(lens[b])
        for h in range(H):
            O[b, h], LSE[b, h] = attention_head(Qf[b, h], Kf[b, h], Vf[b, h], scale, causal, L)
    return O, LSE


def visible_rows(rows, Nq: int, Nk: int, causal: bool, key_len=None) -> np.ndarray:
    """Rows ``rows`` of ``visible``: boolean [len(rows), Nk]."""
    L = Nk if key_len is None else int(min(max(int(key_len), 0), Nk))
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(Nk)[None, :]
    vis = np.broadcast_to(j < L, (i.shape[0], Nk))
    if causal:
        vis = vis & (j <= i + (Nk - Nq))
    return vis


def attention_rows(Q, K, V, scale: float, causal: bool, lens, picks, chunk: int = 1024):
    """Oracle for selected rows only: picks is a list of (b, h, i).

    Every row follows the three-pass definition of ``attention_head`` on its own
    query vector ([FM] "Safe softmax"): s_j = scale * q . k_j with masked keys at
    -inf, m = max s, l = sum exp(s_j - m), O = sum exp(s_j - m) v_j / l,
    LSE = m + ln l; a row with no visible key has O = 0, LSE = -inf.  Rows never
    interact, so the rows of one head are evaluated together, ``chunk`` at a time,
    with that head's keys widened to float64 once; keys past the last key any row
    of the chunk may see are masked for all of them and are left out (they would
    only add exp(-inf) = 0 terms).  This serves problems too large to run whole on
    the CPU.  Returns (O [n, dv], LSE [n]) in the order of ``picks``.
    """
    Nq, Nk = Q.shape[2], K.shape[2]
    dv = V.shape[3]
    O = np.zeros((len(picks), dv))
    LSE = np.full(len(picks), NEG_INF)
    groups = {}
    for r, (b, h, i) in enumerate(picks):
        groups.setdefault((int(b), int(h)), []).append((r, int(i)))
    for (b, h), members in groups.items():
        k = _as_f64(K[b, h])
        v = _as_f64(V[b, h])
        L = None if lens is None else int(lens[b])
        for c0 in range(0, len(members), chunk):
            part = members[c0:c0 + chunk]
            out = np.array([r for r, _ in part], dtype=np.int64)
            rows = np.array([i for _, i in part], dtype=np.int64)
            vis = visible_rows(rows, Nq, Nk, causal, L)
            seen = np.nonzero(vis.any(axis=0))[0]
            kmax = int(seen[-1]) + 1 if seen.size else 0
            if kmax == 0:
                continue                                    # every row fully masked
            q = _as_f64(Q[b, h][rows])
            s = scale * (q @ k[:kmax].T)
            s = np.where(vis[:, :kmax], s, NEG_INF)
            m = s.max(axis=1)                               # pass 1
            live = m > NEG_INF
            ref = np.where(live, m, 0.0)
            p = np.exp(s - ref[:, None])                    # exp(-inf) = 0 for masked keys
            l = p.sum(axis=1)                               # pass 2
            acc = p @ v[:kmax]                              # pass 3
            O[out[live]] = acc[live] / l[live, None]
            LSE[out[live]] = m[live] + np.log(l[live])
    return O, LSE


# --- partial states over a key range, and their merge ---------------------------

def attention_state_head(q, k, v, scale: float, causal: bool, key_len, key_begin: int, key_end: int):
    """The running state (m, l, o~) of every row of one head after absorbing exactly
    the visible keys j with key_begin <= j < key_end, in float64.

    [FM] "The running state": m = max of the scores seen, l = sum exp(s_j - m) and
    o~ = sum exp(s_j - m) v_j over the scores seen (o~ unnormalised).  Written from
    that definition directly (one max, one sum), not through the block loop.  A row
    that saw no visible key in the range has the initial state m = -inf, l = 0, o~ = 0
    ([FM] "The block-wise update, and the full algorithm", init line).

    Returns (o_acc [Nq, dv], m [Nq], l [Nq]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Nq, Nk, dv = q.shape[0], k.shape[0], v.shape[1]
    o_acc = np.zeros((Nq, dv))
    m = np.full(Nq, NEG_INF)
    l = np.zeros(Nq)
    lo, hi = max(int(key_begin), 0), min(int(key_end), Nk)
    if Nq == 0 or hi <= lo:
        return o_acc, m, l
    s = scale * (q @ k[lo:hi].T)
    s = np.where(visible(Nq, Nk, causal, key_len)[:, lo:hi], s, NEG_INF)
    mm = s.max(axis=1)
    live = mm > NEG_INF
    ref = np.where(live, mm, 0.0)
    p = np.exp(s - ref[:, None])
    m[live] = mm[live]
    l[live] = p[live].sum(axis=1)
    o_acc[live] = p[live] @ v[lo:hi]
    return o_acc, m, l


def merge_states(states, _mutation=None):
    """Combine states (o~_s, m_s, l_s) of disjoint key sets into the state of their union.

    Each state is already expressed relative to its own max m_s.  The rescaling
    identity of [FM] "The rescaling identity, derived" moves every one of them to the
    common reference m = max_s m_s with the factor exp(m_s - m) <= 1:
        l = sum_s exp(m_s - m) l_s,   o~ = sum_s exp(m_s - m) o~_s.
    The pages state that keys may be absorbed in any order and in blocks of any size
    ([FM] "The running state"; "Proof of exactness"); a state is such a summary of a
    block, so the identity applies to it as it does to one block.  If every m_s is
    -inf the union saw no visible key: (0, -inf, 0).

    states: list of (o_acc [..., dv], m [...], l [...]).  Returns (o_acc, m, l).
    ``_mutation`` plants a known mistake for the tests that check a pin catches it:
    "rescale_l_only" (o~_s added without its factor) or "no_rescale" (neither l_s nor
    o~_s rescaled).
    """
    if not states:
        raise ValueError("merge_states needs at least one state")
    ms = np.stack([np.asarray(st[1], dtype=np.float64) for st in states])
    m = ms.max(axis=0)
    ref = np.where(m > NEG_INF, m, 0.0)
    o_acc = np.zeros_like(np.asarray(states[0][0], dtype=np.float64))
    l = np.zeros_like(m)
    for o_s, m_s, l_s in states:
        w = np.exp(np.asarray(m_s, dtype=np.float64) - ref)     # exp(-inf) = 0 for an empty state
        wo = w
        if _mutation == "no_rescale":
            w = wo = np.ones_like(w)
        elif _mutation == "rescale_l_only":
            wo = np.ones_like(w)
        l = l + w * np.asarray(l_s, dtype=np.float64)
        o_acc = o_acc + wo[..., None] * np.asarray(o_s, dtype=np.float64)
    return o_acc, m, l


def finish_state(o_acc, m, l):
    """O = o~ / l and LSE = m + ln l: the single final division of [FM] "The block-wise
    update, and the full algorithm"; a state that saw no visible key (l = 0) gives the
    fully masked convention O = 0, LSE = -inf."""
    o_acc = np.asarray(o_acc, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    live = l > 0.0
    O = np.zeros_like(o_acc)
    LSE = np.full(m.shape, NEG_INF)
    O[live] = o_acc[live] / l[live][..., None]
    LSE[live] = m[live] + np.log(l[live])
    return O, LSE


def attention_states(Q, K, V, scale: float, causal: bool, lens, key_ranges):
    """Batched ``attention_state_head`` for a list of key ranges [(begin, end), ...].

    Q [B,H,Nq,d], K/V [B,H,Nk,d] as bf16 codes or floats.  Returns float64
    o_acc [S,B,H,Nq,dv], m [S,B,H,Nq], l [S,B,H,Nq] with S = len(key_ranges).
    """
    Qf, Kf, Vf = (_as_f64(x) for x in (Q, K, V))
    B, H, Nq, _ = Qf.shape
    dv = Vf.shape[3]
    S = len(key_ranges)
    o_acc = np.zeros((S, B, H, Nq, dv))
    m = np.full((S, B, H, Nq), NEG_INF)
    l = np.zeros((S, B, H, Nq))
    for si, (lo, hi) in enumerate(key_ranges):
        for b in range(B):
            L = None if lens is None else int(lens[b])
            for h in range(H):
                o_acc[si, b, h], m[si, b, h], l[si, b, h] = attention_state_head(
                    Qf[b, h], Kf[b, h], Vf[b, h], scale, causal, L, lo, hi)
    return o_acc, m, l


def _as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(np.float64)


# --- the online recurrence, as the pages state it (a second, blockwise route) --

def online_softmax_attention(s, v, block: int, valid=None, order=None, trace=None, _mutation=None):
    """One query row through the block-wise online recurrence, in float64.

    Follows [FM] "The block-wise update, and the full algorithm" and [OS]
    "The Complete Online Softmax Algorithm":

        init  m = -inf, l = 0, o~ = 0
        per block B:  m_blk = max s_B;  m_new = max(m, m_blk);
                      alpha = exp(m - m_new);  p = exp(s_B - m_new);
                      l = alpha*l + sum p;  o~ = alpha*o~ + p.v_B;  m = m_new
        return o~ / l, m, l

    s: raw scores [N]; valid: optional boolean [N], masked keys get -inf
    before the block max ([FM] "Pitfalls"); v: values [N, dv] or [N].
    block: keys per block; order: optional permutation of the block indices.
    trace: optional list that receives a dict per block (m_blk, m, alpha, p, l, o~).
    While m_new is still -inf (every key so far masked) the reference point
    is taken as 0, so alpha = 0 and p = 0 instead of exp(-inf - (-inf)); a row
    with no visible key returns o = 0 (the fully-masked convention).

    ``_mutation`` plants one of the pages' known mistakes, for tests that show
    the pins catch it ([FM] "Pitfalls"; [OS] "The Challenge"):
    "rescale_l_only", "finite_init", "mask_after_max", "normalize_per_block",
    "local_max".
    """
    s = np.asarray(s, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    scalar_v = v.ndim == 1
    if scalar_v:
        v = v[:, None]
    N = s.shape[0]
    if valid is None:
        valid = np.ones(N, dtype=bool)
    valid = np.asarray(valid, dtype=bool)
    masked = np.where(valid, s, NEG_INF)
    nblk = (N + block - 1) // block
    blocks = list(range(nblk)) if order is None else list(order)
    m = 0.0 if _mutation == "finite_init" else NEG_INF
    l = 0.0
    o = np.zeros(v.shape[1])
    for bi in blocks:
        lo, hi = bi * block, min((bi + 1) * block, N)
        sb, vb = masked[lo:hi], v[lo:hi]
        if _mutation == "mask_after_max":
            m_blk = np.max(s[lo:hi])           # max taken over unmasked scores
        else:
            m_blk = np.max(sb)
        if _mutation == "local_max":
            m_new = m_blk                      # each block against its own max
            alpha = 1.0
        else:
            m_new = max(m, m_blk)
            alpha = np.exp(m - (m_new if m_new > NEG_INF else 0.0))
        ref = m_new if m_new > NEG_INF else 0.0
        p = np.exp(sb - ref)
        l = alpha * l + p.sum()
        if _mutation == "rescale_l_only":
            o = o + p @ vb
        elif _mutation == "normalize_per_block":
            o = (alpha * o + p @ vb) / l if l > 0 else o
        else:
            o = alpha * o + p @ vb
        m = m_new
        if trace is not None:
            trace.append(dict(block=bi, m_blk=float(m_blk), m=float(m), alpha=float(alpha), p=p.copy(),
                              l=float(l), o=o.copy()))
    if _mutation == "normalize_per_block":
        out = o
    else:
        out = o / l if l > 0 else np.zeros_like(o)
    return (out[0] if scalar_v else out), m, l
