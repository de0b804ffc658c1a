"""Seeded synthetic inputs for the attention forward, shared by the CUDA path and the oracle.

This module holds no attention arithmetic (no softmax, no exponentials, no
accumulation).  It turns (seed, tensor id, index) into bf16 codes through the
counter-based generator in ``gen.c`` and builds the workloads below.  The only
arithmetic beyond sampling is the planting of a chosen score in the
adversarial workload, which needs one dot product per row to place it.

bf16 tensors are returned as ``numpy.uint16`` arrays of raw codes, layout
``[B, H, N, d]`` row-major.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_gen.so")
_lock = threading.Lock()
_lib = None

# tensor ids of the streams drawn from one seed
TID_Q, TID_K, TID_V, TID_LENS, TID_PLANT = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile gen.c into _gen.so beside it (portable C99, gcc)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", _SRC, "-o", tmp, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            i32p = ctypes.POINTER(ctypes.c_int32)
            u64p = ctypes.POINTER(ctypes.c_uint64)
            lib.gen_normal_bf16.argtypes = [u16p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                            ctypes.c_double, ctypes.c_double, ctypes.c_int]
            lib.gen_uniform_bf16.argtypes = lib.gen_normal_bf16.argtypes
            lib.gen_uniform_int.argtypes = [i32p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                            ctypes.c_int32, ctypes.c_int32]
            lib.gen_raw_u64.argtypes = [u64p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32]
            lib.gen_splitmix64_sequence.argtypes = [u64p, ctypes.c_int64, ctypes.c_uint64]
            for f in (lib.gen_normal_bf16, lib.gen_uniform_bf16, lib.gen_uniform_int, lib.gen_raw_u64,
                      lib.gen_splitmix64_sequence):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def normal_bf16(shape, seed: int, tensor_id: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    rc = _load().gen_normal_bf16(_ptr(out, ctypes.c_uint16), out.size, seed, tensor_id, mu, sigma, _threads())
    if rc != 0:
        raise RuntimeError("gen_normal_bf16 failed")
    return out


def uniform_bf16(shape, seed: int, tensor_id: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    rc = _load().gen_uniform_bf16(_ptr(out, ctypes.c_uint16), out.size, seed, tensor_id, lo, hi, _threads())
    if rc != 0:
        raise RuntimeError("gen_uniform_bf16 failed")
    return out


def uniform_int(n: int, seed: int, tensor_id: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    rc = _load().gen_uniform_int(_ptr(out, ctypes.c_int32), n, seed, tensor_id, lo, hi)
    if rc != 0:
        raise RuntimeError("gen_uniform_int failed")
    return out


def raw_u64(n: int, seed: int, tensor_id: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().gen_raw_u64(_ptr(out, ctypes.c_uint64), n, seed, tensor_id)
    return out


def splitmix64_sequence(n: int, seed: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().gen_splitmix64_sequence(_ptr(out, ctypes.c_uint64), n, seed)
    return out


# --- bf16 code <-> float conversion used only to build inputs -----------------

def codes_to_f32(codes: np.ndarray) -> np.ndarray:
    return (np.asarray(codes, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_codes(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 codes, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# --- workloads ----------------------------------------------------------------

class Workload(dict):
    """Shape, mask and value recipe of one synthetic attention problem."""

    @property
    def name(self) -> str:
        return self["name"]


def _wl(**kw) -> Workload:
    w = Workload(kw)
    w.setdefault("Nk", w["Nq"])
    w.setdefault("lens", None)
    w.setdefault("plant", None)
    w.setdefault("scale", 1.0 / math.sqrt(w["d"]))
    return w


WORKLOADS = {
    w.name: w
    for w in [
        _wl(name="b1h2n256d64", B=1, H=2, Nq=256, d=64, causal=False, qk=("normal", 0.0, 1.0),
            v=("normal", 0.0, 1.0), seed=1001),
        _wl(name="causal_b4h16n2048d128", B=4, H=16, Nq=2048, d=128, causal=True, qk=("normal", 0.0, 1.0),
            v=("normal", 0.0, 1.0), seed=1002),
        _wl(name="causal_b2h32n8192d128", B=2, H=32, Nq=8192, d=128, causal=True, qk=("normal", 0.0, 1.0),
            v=("normal", 0.0, 1.0), seed=1003),
        # planted maxima (score ~ +60) in the first key tile for even rows and in the
        # last valid key tile for odd rows; V uniform in [-100, 100]; key padding with
        # batch 0 fully masked (length 0) and batch 1 uniform in [1, 4095].
        _wl(name="padded_planted_b2h8n4096d128", B=2, H=8, Nq=4096, d=128, causal=False,
            qk=("normal", 0.0, 1.0), v=("uniform", -100.0, 100.0), lens=("fixed0_then_uniform", 1, 4095),
            plant=dict(score=60.0, tile=128), seed=1004),
        _wl(name="causal_b1h32n32768d128", B=1, H=32, Nq=32768, d=128, causal=True, qk=("normal", 0.0, 0.5),
            v=("normal", 0.0, 0.5), seed=1005),
        _wl(name="causal_b1h32n32768d64", B=1, H=32, Nq=32768, d=64, causal=True, qk=("normal", 0.0, 0.5),
            v=("normal", 0.0, 0.5), seed=1006),
        # few query rows over a long key sequence (decoding a chunk of 128 tokens against a
        # 32K cache, bottom-right causal): 32 query tiles for 152 SMs, the split-KV shape
        _wl(name="causal_b1h32q128k32768d128", B=1, H=32, Nq=128, Nk=32768, d=128, causal=True,
            qk=("normal", 0.0, 0.5), v=("normal", 0.0, 0.5), seed=1007),
    ]
}


def _draw(kind, shape, seed, tid):
    if kind[0] == "normal":
        return normal_bf16(shape, seed, tid, kind[1], kind[2])
    if kind[0] == "uniform":
        return uniform_bf16(shape, seed, tid, kind[1], kind[2])
    raise ValueError(kind)


def make_lens(w: Workload):
    spec = w["lens"]
    if spec is None:
        return None
    if spec[0] == "fixed0_then_uniform":
        lens = uniform_int(w["B"], w["seed"], TID_LENS, spec[1], spec[2])
        lens[0] = 0
        return lens
    if spec[0] == "given":
        return np.asarray(spec[1], dtype=np.int32)
    raise ValueError(spec)


def plant_scores(Q: np.ndarray, K: np.ndarray, lens, scale: float, score: float, tile: int, seed: int):
    """Move each query row so that its score with one chosen key is ``score``.

    Even rows take the key from the first key tile, odd rows from the last
    valid tile [max(0, L_b - tile), L_b).  q_i <- q_i + beta * k_j with beta set
    in float64 from the bf16 values so that scale * q_i . k_j equals ``score``
    before q_i is rounded back to bf16.  Rows of a batch with no valid key are
    left unchanged.  Returns the new Q codes and the chosen key index per row.
    """
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    u = raw_u64(B * H * Nq, seed, TID_PLANT).reshape(B, H, Nq)
    u = (u >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    Qn = Q.copy()
    jstar = np.full((B, H, Nq), -1, dtype=np.int64)
    rows = np.arange(Nq)
    for b in range(B):
        L = Nk if lens is None else int(min(max(lens[b], 0), Nk))
        if L == 0:
            continue
        first_lo, first_hi = 0, min(tile, L)
        last_lo, last_hi = max(0, L - tile), L
        lo = np.where(rows % 2 == 0, first_lo, last_lo)
        hi = np.where(rows % 2 == 0, first_hi, last_hi)
        for h in range(H):
            j = lo + np.floor(u[b, h] * (hi - lo)).astype(np.int64)
            j = np.minimum(j, hi - 1)
            q = codes_to_f32(Q[b, h]).astype(np.float64)
            k = codes_to_f32(K[b, h, j]).astype(np.float64)
            qk = np.einsum("nd,nd->n", q, k)
            kk = np.einsum("nd,nd->n", k, k)
            beta = (score / scale - qk) / kk
            Qn[b, h] = f32_to_codes((q + beta[:, None] * k).astype(np.float32))
            jstar[b, h] = j
    return Qn, jstar


def make_inputs(w, **override) -> dict:
    """Generate one workload's tensors: dict(Q, K, V, lens, scale, causal, ...)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    w = Workload({**w, **override})
    B, H, Nq, Nk, d = w["B"], w["H"], w["Nq"], w["Nk"], w["d"]
    seed = w["seed"]
    Q = _draw(w["qk"], (B, H, Nq, d), seed, TID_Q)
    K = _draw(w["qk"], (B, H, Nk, d), seed, TID_K)
    V = _draw(w["v"], (B, H, Nk, d), seed, TID_V)
    lens = make_lens(w)
    out = dict(Q=Q, K=K, V=V, lens=lens, scale=float(w["scale"]), causal=bool(w["causal"]), B=B, H=H, Nq=Nq,
               Nk=Nk, d=d, name=w.get("name", "custom"))
    if w.get("plant"):
        p = w["plant"]
        out["Q"], out["planted_key"] = plant_scores(Q, K, lens, w["scale"], p["score"], p["tile"], seed)
    return out



# --- packed sequences of different lengths --------------------------------------

VARLEN_WORKLOADS = {
    # 16 prompts of 512..8192 tokens (seeded uniform), 16 heads, d = 128, causal within
    # each prompt, N(0, 1) values, packed row after row: [total, H, d]
    "varlen_causal_b16h16d128": dict(name="varlen_causal_b16h16d128", B=16, H=16, d=128, causal=True,
                                     lengths=("uniform", 512, 8192), qk=("normal", 0.0, 1.0),
                                     v=("normal", 0.0, 1.0), seed=1008),
}


def make_varlen(name: str) -> dict:
    """Packed inputs: Q, K, V codes [total, H, d], cu [B + 1] (the same for queries and
    keys), lengths, scale, causal."""
    w = VARLEN_WORKLOADS[name]
    lo, hi = w["lengths"][1], w["lengths"][2]
    lengths = uniform_int(w["B"], w["seed"], TID_LENS, lo, hi).astype(np.int64)
    total = int(lengths.sum())
    shape = (total, w["H"], w["d"])
    Q = _draw(w["qk"], shape, w["seed"], TID_Q)
    K = _draw(w["qk"], shape, w["seed"], TID_K)
    V = _draw(w["v"], shape, w["seed"], TID_V)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return dict(name=name, Q=Q, K=K, V=V, cu=cu, lengths=lengths, total=total, B=w["B"], H=w["H"], d=w["d"],
                causal=w["causal"], scale=1.0 / math.sqrt(w["d"]))
