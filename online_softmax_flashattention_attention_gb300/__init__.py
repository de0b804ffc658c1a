"""Python binding of the fused attention forward library (``libattn.so``, C ABI in include/attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing or a call fails, an exception is
raised.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

EXPORTS = ("attn_fwd", "attn_fwd_ex", "attn_fwd_strided", "attn_fwd_varlen", "attn_fwd_host", "attn_release_workspace", "attn_status_sync", "attn_last_error",
           "attn_version", "attn_fwd_noalloc", "attn_fwd_states", "attn_merge_states",
           "attn_splitkv_workspace_bytes", "attn_splitkv_splits", "attn_fwd_splitkv")

STATUS_NAMES = {0: "ATTN_OK", -1: "ATTN_ERR_NULLPTR", -2: "ATTN_ERR_BAD_SHAPE", -3: "ATTN_ERR_UNSUPPORTED_D",
                -4: "ATTN_ERR_MISALIGNED", -5: "ATTN_ERR_NO_DEVICE", -6: "ATTN_ERR_LAUNCH", -7: "ATTN_ERR_TIMEOUT",
                -8: "ATTN_ERR_BAD_ARG"}


EXP2_DEFAULT, EXP2_HARDWARE, EXP2_MIXED = 0, 1, 2


class AttnOptions(ctypes.Structure):
    """attn_options of include/attn.h."""
    _fields_ = [("size", ctypes.c_size_t), ("rescale_threshold", ctypes.c_float), ("exp2_mode", ctypes.c_int),
                ("key_block", ctypes.c_int)]


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library():
    """Load libattn.so (built by ``__graft_entry__.build()``); raises if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        sig = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp]
        for name in ("attn_fwd", "attn_fwd_host"):
            getattr(lib, name).argtypes = sig
            getattr(lib, name).restype = i
        lib.attn_release_workspace.argtypes = []
        lib.attn_release_workspace.restype = i
        lib.attn_status_sync.argtypes = [vp]
        lib.attn_status_sync.restype = i
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_version.argtypes = []
        lib.attn_version.restype = i
        lib.attn_fwd_ex.argtypes = sig[:-1] + [ctypes.POINTER(AttnOptions), vp]
        lib.attn_fwd_ex.restype = i
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.attn_fwd_strided.argtypes = sig[:-1] + [i64p, i64p, i64p, i64p, vp]
        lib.attn_fwd_strided.restype = i
        lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.attn_fwd_varlen.restype = i
        lib.attn_fwd_states.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp]
        lib.attn_fwd_states.restype = i
        lib.attn_merge_states.argtypes = [vp, vp, vp, i, ctypes.c_longlong, i, vp, vp, vp]
        lib.attn_merge_states.restype = i
        lib.attn_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_splitkv_splits.argtypes = [i, i, i, i]
        lib.attn_splitkv_splits.restype = i
        lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, ctypes.c_size_t, vp]
        lib.attn_fwd_splitkv.restype = i
        _lib = lib
    return _lib


def _check(rc: int):
    if rc != 0:
        raise AttnError(rc, load_library().attn_last_error().decode())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def attn_fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale, causal, lens_ptr, stream_ptr) -> int:
    """The C call with plain integers for pointers; returns the attn_status code."""
    lib = load_library()
    return lib.attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale, int(causal), lens_ptr,
                        stream_ptr)


def _check_qkv(Q, K, V, key_padding_lens):
    """Shapes, dtypes and placement of the inputs; returns (B, H, Nq, Nk, d, lens_ptr)."""
    import torch
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if K.shape != (B, H, Nk, d) or V.shape != (B, H, Nk, d):
        raise ValueError("K and V must be [B, H, Nk, d] with Q's B, H and d")
    lens_ptr = None
    if key_padding_lens is not None:
        if key_padding_lens.dtype != torch.int32 or not key_padding_lens.is_cuda or key_padding_lens.numel() != B:
            raise ValueError("key_padding_lens must be an int32 CUDA tensor [B]")
        lens_ptr = key_padding_lens.data_ptr()
    return B, H, Nq, Nk, d, lens_ptr


def _outputs(Q, O, LSE):
    import torch
    B, H, Nq, _ = Q.shape
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    if O.shape != Q.shape or O.dtype != torch.bfloat16 or not O.is_contiguous():
        raise ValueError("O must be a contiguous bf16 tensor shaped like Q")
    if LSE.shape != (B, H, Nq) or LSE.dtype != torch.float32 or not LSE.is_contiguous():
        raise ValueError("LSE must be a contiguous fp32 tensor [B, H, Nq]")
    return O, LSE


def attn_fwd(Q, K, V, O=None, LSE=None, *, scale=None, causal=False, key_padding_lens=None, stream=None,
             rescale_threshold=0.0, exp2_mode=EXP2_DEFAULT, key_block=0):
    """O, LSE = softmax(scale * Q K^T + mask) V and its row logsumexp, on the GPU.

    Q [B,H,Nq,d], K/V [B,H,Nk,d]: contiguous bf16 CUDA tensors.  O (bf16) and LSE
    (fp32 [B,H,Nq]) are allocated when not given.  key_padding_lens: int32 CUDA
    tensor [B] or None.  Enqueued on ``stream`` (default: torch's current stream).
    rescale_threshold / exp2_mode / key_block: the attn_options of attn_fwd_ex (defaults:
    attn_fwd).
    """
    import torch
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if K.shape != (B, H, Nk, d) or V.shape != (B, H, Nk, d):
        raise ValueError("K and V must be [B, H, Nk, d] with Q's B, H and d")
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    if O.shape != Q.shape or O.dtype != torch.bfloat16 or not O.is_contiguous():
        raise ValueError("O must be a contiguous bf16 tensor shaped like Q")
    if LSE.shape != (B, H, Nq) or LSE.dtype != torch.float32 or not LSE.is_contiguous():
        raise ValueError("LSE must be a contiguous fp32 tensor [B, H, Nq]")
    lens_ptr = None
    if key_padding_lens is not None:
        if key_padding_lens.dtype != torch.int32 or not key_padding_lens.is_cuda or key_padding_lens.numel() != B:
            raise ValueError("key_padding_lens must be an int32 CUDA tensor [B]")
        lens_ptr = key_padding_lens.data_ptr()
    if rescale_threshold == 0.0 and exp2_mode == EXP2_DEFAULT and key_block == 0:
        rc = attn_fwd_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H, Nq, Nk, d,
                          float(scale), causal, lens_ptr, _stream_handle(stream))
    else:
        opts = AttnOptions(ctypes.sizeof(AttnOptions), float(rescale_threshold), int(exp2_mode), int(key_block))
        rc = load_library().attn_fwd_ex(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H,
                                        Nq, Nk, d, float(scale), int(causal), lens_ptr, ctypes.byref(opts),
                                        _stream_handle(stream))
    _check(rc)
    return O, LSE


def attn_fwd_host(Q, K, V, O, LSE, *, scale=None, causal=False, key_padding_lens=None, stream=None):
    """Host-buffer variant: Q/K/V/O are CPU bf16 tensors (pinned for speed), LSE CPU fp32,
    key_padding_lens a CPU int32 tensor or None.  Blocks until O and LSE are written."""
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lens_ptr = None if key_padding_lens is None else key_padding_lens.data_ptr()
    lib = load_library()
    rc = lib.attn_fwd_host(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H, Nq, Nk, d,
                           float(scale), int(causal), lens_ptr, _stream_handle(stream))
    _check(rc)
    return O, LSE


def status_sync(stream=None):
    """Synchronise the stream and raise AttnError if a bounded device wait ran out."""
    _check(load_library().attn_status_sync(_stream_handle(stream)))


def release_workspace():
    _check(load_library().attn_release_workspace())


def version() -> int:
    return load_library().attn_version()


# --- split-KV: partial states and their merge ---------------------------------

def attn_fwd_states(Q, K, V, num_splits, *, scale=None, causal=False, key_padding_lens=None, stream=None):
    """The running states (o~, m, l) of ``num_splits`` key splits (split s covers keys
    [s*C, (s+1)*C), C = 128 * ceil(ceil(Nk/128) / num_splits)).  Returns fp32 CUDA tensors
    o_states [S,B,H,Nq,d], m_states [S,B,H,Nq], l_states [S,B,H,Nq]."""
    import torch
    B, H, Nq, Nk, d, lens_ptr = _check_qkv(Q, K, V, key_padding_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    S = int(num_splits)
    o_st = torch.empty((S, B, H, Nq, d), dtype=torch.float32, device=Q.device)
    m_st = torch.empty((S, B, H, Nq), dtype=torch.float32, device=Q.device)
    l_st = torch.empty((S, B, H, Nq), dtype=torch.float32, device=Q.device)
    rc = load_library().attn_fwd_states(Q.data_ptr(), K.data_ptr(), V.data_ptr(), o_st.data_ptr(), m_st.data_ptr(),
                                        l_st.data_ptr(), B, H, Nq, Nk, d, float(scale), int(causal), lens_ptr, S,
                                        _stream_handle(stream))
    _check(rc)
    return o_st, m_st, l_st


def merge_states(o_states, m_states, l_states, O=None, LSE=None, *, stream=None):
    """Merge S states per row: o_states fp32 [S, ..., d], m_states / l_states fp32 [S, ...].
    Returns O bf16 [..., d] and LSE fp32 [...] (allocated when not given)."""
    import torch
    S, d = o_states.shape[0], o_states.shape[-1]
    rows_shape = tuple(o_states.shape[1:-1])
    for name, t in (("o_states", o_states), ("m_states", m_states), ("l_states", l_states)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    if tuple(m_states.shape) != (S,) + rows_shape or tuple(l_states.shape) != (S,) + rows_shape:
        raise ValueError("m_states and l_states must be [S, ...] matching o_states [S, ..., d]")
    if O is None:
        O = torch.empty(rows_shape + (d,), dtype=torch.bfloat16, device=o_states.device)
    if LSE is None:
        LSE = torch.empty(rows_shape, dtype=torch.float32, device=o_states.device)
    rows = int(math.prod(rows_shape))
    if O.numel() != rows * d or O.dtype != torch.bfloat16 or LSE.numel() != rows or LSE.dtype != torch.float32:
        raise ValueError("O must be bf16 [..., d] and LSE fp32 [...] over the states' rows")
    rc = load_library().attn_merge_states(o_states.data_ptr(), m_states.data_ptr(), l_states.data_ptr(), S, rows, d,
                                          O.data_ptr(), LSE.data_ptr(), _stream_handle(stream))
    _check(rc)
    return O, LSE


def splitkv_splits(B, H, Nq, Nk) -> int:
    """The split count attn_fwd_splitkv picks for num_splits <= 0 on the current device."""
    return load_library().attn_splitkv_splits(B, H, Nq, Nk)


def splitkv_workspace_bytes(B, H, Nq, d, num_splits) -> int:
    return load_library().attn_splitkv_workspace_bytes(B, H, Nq, d, num_splits)


def attn_fwd_splitkv(Q, K, V, O=None, LSE=None, *, num_splits=0, workspace=None, scale=None, causal=False,
                     key_padding_lens=None, stream=None):
    """attn_fwd through split-KV states and their merge.  workspace: a CUDA uint8 tensor
    of at least splitkv_workspace_bytes(...) bytes, allocated here when not given."""
    import torch
    B, H, Nq, Nk, d, lens_ptr = _check_qkv(Q, K, V, key_padding_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O, LSE = _outputs(Q, O, LSE)
    S = int(num_splits) if num_splits and num_splits > 0 else splitkv_splits(B, H, Nq, Nk)
    need = splitkv_workspace_bytes(B, H, Nq, d, S) if S > 1 else 0
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().attn_fwd_splitkv(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H,
                                         Nq, Nk, d, float(scale), int(causal), lens_ptr, S, ws_ptr, ws_bytes,
                                         _stream_handle(stream))
    _check(rc)
    return O, LSE


# --- other layouts -------------------------------------------------------------

def attn_fwd_strided(Q, K, V, O=None, LSE=None, *, scale=None, causal=False, key_padding_lens=None, stream=None):
    """attn_fwd on 4-D bf16 CUDA tensors viewed as [B, H, N, d] with any strides whose last
    dimension is contiguous (e.g. ``x.transpose(1, 2)`` of a [B, N, H, d] tensor).  O (same
    strides as a new tensor shaped like Q's view when not given) and LSE [B, H, Nq]."""
    import torch
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.stride(3) != 1:
            raise ValueError(f"{name} must be a bf16 CUDA tensor with a contiguous last dimension")
    if K.shape != (B, H, Nk, d) or V.shape != (B, H, Nk, d):
        raise ValueError("K and V must be [B, H, Nk, d] with Q's B, H and d")
    if O is None:
        O = torch.empty((B, Nq, H, d), dtype=torch.bfloat16, device=Q.device).transpose(1, 2)
    if LSE is None:
        LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    if O.shape != Q.shape or O.dtype != torch.bfloat16 or O.stride(3) != 1:
        raise ValueError("O must be bf16 shaped like Q with a contiguous last dimension")
    lens_ptr = None
    if key_padding_lens is not None:
        lens_ptr = key_padding_lens.data_ptr()

    def st(t):
        return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))
    rc = load_library().attn_fwd_strided(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H,
                                         Nq, Nk, d, float(scale), int(causal), lens_ptr, st(Q), st(K), st(V), st(O),
                                         _stream_handle(stream))
    _check(rc)
    return O, LSE


def attn_fwd_varlen(Q, K, V, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, O=None, LSE=None, *, scale=None, causal=False,
                    stream=None):
    """Packed sequences: Q [total_q, H, d], K/V [total_k, H, d] contiguous bf16 CUDA tensors,
    cu_seqlens_q / cu_seqlens_k int32 CUDA tensors [B + 1].  Returns O [total_q, H, d] and
    LSE [H, total_q]."""
    import torch
    total_q, H, d = Q.shape
    total_k = K.shape[0]
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((H, total_q), dtype=torch.float32, device=Q.device)
    rc = load_library().attn_fwd_varlen(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                                        cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, H, int(max_seqlen_q),
                                        total_q, total_k, d, float(scale), int(causal), _stream_handle(stream))
    _check(rc)
    return O, LSE


# --- the CPU library (libattn_cpu.so, include/attn_cpu.h) ------------------------

CPU_LIB_PATH = os.path.join(_HERE, "libattn_cpu.so")
CPU_EXPORTS = ("attn_fwd_cpu",)
_cpu_lib = None


def load_cpu_library():
    """Load libattn_cpu.so (built by __graft_entry__.build()); raises if it is absent."""
    global _cpu_lib
    if _cpu_lib is None:
        if not os.path.exists(CPU_LIB_PATH):
            raise ImportError(f"{CPU_LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(CPU_LIB_PATH)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd_cpu.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, i]
        lib.attn_fwd_cpu.restype = i
        _cpu_lib = lib
    return _cpu_lib


def attn_fwd_cpu(Q, K, V, *, scale=None, causal=False, key_padding_lens=None, num_threads=0):
    """The forward on the host CPU.  Q [B,H,Nq,d], K/V [B,H,Nk,d]: numpy uint16 arrays of
    bf16 codes.  Returns O (uint16 codes, same shape as Q) and LSE (float32 [B,H,Nq])."""
    import numpy as np
    Q, K, V = (np.ascontiguousarray(a, dtype=np.uint16) for a in (Q, K, V))
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if K.shape != (B, H, Nk, d) or V.shape != (B, H, Nk, d):
        raise ValueError("K and V must be [B, H, Nk, d] with Q's B, H and d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.empty_like(Q)
    LSE = np.empty((B, H, Nq), dtype=np.float32)
    lens = None if key_padding_lens is None else np.ascontiguousarray(key_padding_lens, dtype=np.int32)
    rc = load_cpu_library().attn_fwd_cpu(Q.ctypes.data, K.ctypes.data if Nk else None, V.ctypes.data if Nk else None,
                                         O.ctypes.data, LSE.ctypes.data, B, H, Nq, Nk, d, float(scale), int(causal),
                                         None if lens is None else lens.ctypes.data, int(num_threads))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_cpu failed")
    return O, LSE
