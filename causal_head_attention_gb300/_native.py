"""ctypes binding of librca_attn.so: the C ABI in include/rca_attn.h, same names.

Argument marshalling only: tensors are turned into device pointers and sizes,
and every step of the computation runs in the library's CUDA kernels. There is
no CPU fallback: if the library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "librca_attn.so")

RCA_OK = 0
RCA_ERR_INVALID_ARGUMENT = 1
RCA_ERR_UNSUPPORTED = 2
RCA_ERR_CUDA = 3
RCA_ERR_DEVICE_TIMEOUT = 4
RCA_ERR_DEVICE_INVALID_INPUT = 5
RCA_F32_TF32 = 0
RCA_BF16 = 1

STATUS_NAMES = {
    0: "RCA_OK",
    1: "RCA_ERR_INVALID_ARGUMENT",
    2: "RCA_ERR_UNSUPPORTED",
    3: "RCA_ERR_CUDA",
    4: "RCA_ERR_DEVICE_TIMEOUT",
    5: "RCA_ERR_DEVICE_INVALID_INPUT",
}

# Every symbol include/rca_attn.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int64
_SIG = {
    "rca_abi_version": (ctypes.c_uint32, []),
    "rca_last_error": (ctypes.c_char_p, []),
    "rca_attn_fwd": (ctypes.c_int, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, ctypes.c_int, _P]),
    "rca_attn_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, ctypes.c_int]),
    "rca_attn_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                    ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "rca_attn_bwd_preprocess": (ctypes.c_int, [_P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_int, _P,
                                               ctypes.c_size_t, _P]),
    "rca_attn_bwd_main": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_int,
                                         _P, ctypes.c_size_t, _P]),
    "rca_attn_bwd_dq_convert": (ctypes.c_int, [_P, _I, _I, _I, _I, _I, ctypes.c_int, _P,
                                               ctypes.c_size_t, _P]),
    "rca_attn_bwd_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                            ctypes.c_int, _P]),
    "rca_paged_decode_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, ctypes.c_int]),
    "rca_paged_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_int,
                                        _P, ctypes.c_size_t, _P]),
    "rca_attn_materialized_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, ctypes.c_int]),
    "rca_attn_materialized_fwd": (ctypes.c_int, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, ctypes.c_int, _P,
                                                 ctypes.c_size_t, _P]),
    "rca_attn_materialized_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                                 ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "rca_causal_softmax": (ctypes.c_int, [_P, _P, _I, _I, ctypes.c_float, _P]),
    "rca_causal_softmax_bwd": (ctypes.c_int, [_P, _P, _P, _I, _I, ctypes.c_float, _P]),
    "rca_causal_softmax_bwd_tiled": (ctypes.c_int, [_P, _P, _P, _I, _I, _I, ctypes.c_float, _P]),
    "rca_attn_fwd_qkv": (ctypes.c_int, [_P, _I, _I, _I, _I, _I, _P, _P, ctypes.c_int, _P]),
    "rca_attn_bwd_qkv": (ctypes.c_int, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_int, _P, ctypes.c_size_t,
                                        _P]),
    "rca_attn_varlen_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, ctypes.c_int]),
    "rca_attn_fwd_varlen": (ctypes.c_int, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, ctypes.c_int, _P,
                                           ctypes.c_size_t, _P]),
    "rca_attn_bwd_varlen": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                           ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "rca_selftest_device_timeout": (ctypes.c_int, [_P]),
    "rca_selftest_noalloc_timeout": (ctypes.c_int, [_P]),
    "rca_stream_status": (ctypes.c_int, [_P]),
    "rca_set_wait_timeout_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
}

_lib = None


class RcaError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


def lib() -> ctypes.CDLL:
    """Load librca_attn.so (built in-tree by causal_head_attention_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m causal_head_attention_gb300.build` "
                "(the CUDA library is the only implementation; there is no fallback)"
            )
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(status: int):
    if status != RCA_OK:
        raise RcaError(status, lib().rca_last_error().decode(errors="replace"))


# ---------------------------------------------------------------------------
# torch-tensor marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return RCA_BF16
    if t.dtype == torch.float32:
        return RCA_F32_TF32
    raise TypeError(f"unsupported dtype {t.dtype}: expected torch.bfloat16 or torch.float32")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("all tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("all tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _shape(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B,T,Hq,Dh] and k, v [B,T,Hkv,Dh]")
    B, T, Hq, Dh = q.shape
    return B, Hq, k.shape[2], T, Dh


def _attn_args(q, k, v=None, *, like_q=(), like_k=(), lse=None, workspace=None):
    """Checks every tensor of a full-sequence call against q and k before any
    pointer reaches the library: q [B,T,Hq,Dh], k and v [B,T,Hkv,Dh] with the
    same B, T and Dh; the tensors in like_q (out, dout, dq) shaped and typed as
    q, those in like_k (dk, dv) as k; lse float32 [B,Hq,T]; all on q's device.
    Returns (B, Hq, Hkv, T, Dh)."""
    torch = _torch()
    B, Hq, Hkv, T, Dh = _shape(q, k)
    if tuple(k.shape) != (B, T, Hkv, Dh):
        raise ValueError(f"k must be [B,T,Hkv,Dh] with q's B, T and Dh; got q {tuple(q.shape)}, k {tuple(k.shape)}")
    named = [("k", k, (B, T, Hkv, Dh))]
    if v is not None:
        named.append(("v", v, (B, T, Hkv, Dh)))
    named += [(n, t, (B, T, Hq, Dh)) for n, t in like_q]
    named += [(n, t, (B, T, Hkv, Dh)) for n, t in like_k]
    for name, t, shape in named:
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have q's dtype {q.dtype}, got {t.dtype}")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    if lse is not None:
        if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, T):
            raise ValueError(f"lse must be float32 [B,Hq,T] = {(B, Hq, T)}, got {lse.dtype} {tuple(lse.shape)}")
        if lse.device != q.device:
            raise ValueError(f"lse is on {lse.device}, q on {q.device}")
    if workspace is not None and workspace.device != q.device:
        raise ValueError(f"workspace is on {workspace.device}, q on {q.device}")
    return B, Hq, Hkv, T, Dh


def rca_abi_version() -> int:
    return lib().rca_abi_version()


def rca_last_error() -> str:
    return lib().rca_last_error().decode(errors="replace")


def rca_set_wait_timeout_ns(ns: int) -> int:
    return lib().rca_set_wait_timeout_ns(ns)


def rca_attn_fwd(q, k, v, out, lse, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("out", out)], lse=lse)
    _check(lib().rca_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, T, Dh, _ptr(out), _ptr(lse),
                              _dtype_code(q), _stream(stream)))


def rca_attn_bwd_workspace_size(B, Hq, Hkv, T, Dh, dt) -> int:
    """dt: RCA_BF16 / RCA_F32_TF32, or a torch dtype."""
    if not isinstance(dt, int):
        torch = _torch()
        dt = RCA_BF16 if dt == torch.bfloat16 else RCA_F32_TF32
    return lib().rca_attn_bwd_workspace_size(B, Hq, Hkv, T, Dh, dt)


def rca_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, workspace, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("out", out), ("dout", dout), ("dq", dq)],
                                   like_k=[("dk", dk), ("dv", dv)], lse=lse, workspace=workspace)
    _check(lib().rca_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, Hq, Hkv, T, Dh, _dtype_code(q), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)))


def rca_attn_bwd_preprocess(out, lse, dout, workspace, Hkv=None, stream=None):
    _attn_args(out, out, like_q=[("dout", dout)], lse=lse, workspace=workspace)
    B, T, Hq, Dh = out.shape
    Hkv = Hq if Hkv is None else Hkv
    _check(lib().rca_attn_bwd_preprocess(_ptr(out), _ptr(lse), _ptr(dout), B, Hq, Hkv, T, Dh, _dtype_code(out),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def rca_attn_bwd_main(q, k, v, dout, dk, dv, workspace, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("dout", dout)], like_k=[("dk", dk), ("dv", dv)],
                                   workspace=workspace)
    _check(lib().rca_attn_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dk), _ptr(dv), B, Hq, Hkv, T,
                                   Dh, _dtype_code(q), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def rca_attn_bwd_dq_convert(dq, workspace, Hkv=None, stream=None):
    B, T, Hq, Dh = dq.shape
    Hkv = Hq if Hkv is None else Hkv
    _check(lib().rca_attn_bwd_dq_convert(_ptr(dq), B, Hq, Hkv, T, Dh, _dtype_code(dq), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))


def rca_attn_bwd_noalloc(q, k, v, out, lse, dout, dq, dk, dv, stream=None):
    """Backward with the library's built-in scratch (no workspace, no allocation)."""
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("out", out), ("dout", dout), ("dq", dq)],
                                   like_k=[("dk", dk), ("dv", dv)], lse=lse)
    _check(lib().rca_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                      _ptr(dk), _ptr(dv), B, Hq, Hkv, T, Dh, _dtype_code(q), _stream(stream)))


def rca_paged_decode_workspace_size(B, Hq, Hkv, Dh, page_size, max_pages, dt) -> int:
    """dt: RCA_BF16 / RCA_F32_TF32, or a torch dtype."""
    if not isinstance(dt, int):
        torch = _torch()
        dt = RCA_BF16 if dt == torch.bfloat16 else RCA_F32_TF32
    return lib().rca_paged_decode_workspace_size(B, Hq, Hkv, Dh, page_size, max_pages, dt)


def rca_paged_decode(q, k_pool, v_pool, page_table, seq_lens, out, lse, workspace, stream=None):
    """q, out [B,Hq,Dh]; k_pool, v_pool [P,Hkv,page_size,Dh]; page_table [B,max_pages]
    int32; seq_lens [B] int32; lse [B,Hq] float32; workspace a device buffer of at
    least rca_paged_decode_workspace_size(...) bytes."""
    torch = _torch()
    if q.dim() != 3 or k_pool.dim() != 4 or page_table.dim() != 2:
        raise ValueError("q must be [B,Hq,Dh], the pools [P,Hkv,page_size,Dh], page_table [B,max_pages]")
    if page_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("page_table and seq_lens must be int32")
    B, Hq, Dh = q.shape
    P, Hkv, page_size, _ = k_pool.shape
    if (tuple(v_pool.shape) != tuple(k_pool.shape) or k_pool.shape[3] != Dh or tuple(out.shape) != (B, Hq, Dh)
            or tuple(lse.shape) != (B, Hq) or tuple(seq_lens.shape) != (B,) or page_table.shape[0] != B):
        raise ValueError("inconsistent shapes: q, out [B,Hq,Dh]; k_pool, v_pool [P,Hkv,page_size,Dh]; "
                         "page_table [B,max_pages]; seq_lens [B]; lse [B,Hq]")
    if k_pool.dtype != q.dtype or v_pool.dtype != q.dtype or out.dtype != q.dtype or lse.dtype != torch.float32:
        raise TypeError("q, k_pool, v_pool and out share the storage dtype; lse is float32")
    _check(lib().rca_paged_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), B, Hq,
                                  Hkv, Dh, page_size, page_table.shape[1], P, _ptr(out), _ptr(lse),
                                  _dtype_code(q), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def rca_attn_materialized_workspace_size(B, Hq, Hkv, T, Dh, dt) -> int:
    """dt: RCA_BF16 / RCA_F32_TF32, or a torch dtype."""
    if not isinstance(dt, int):
        torch = _torch()
        dt = RCA_BF16 if dt == torch.bfloat16 else RCA_F32_TF32
    return lib().rca_attn_materialized_workspace_size(B, Hq, Hkv, T, Dh, dt)


def _check_probs(probs, B, Hq, T, name="probs"):
    torch = _torch()
    if probs.dtype != torch.float32 or tuple(probs.shape) != (B, Hq, T, T):
        raise ValueError(f"{name} must be float32 [B,Hq,T,T] = {(B, Hq, T, T)}")


def rca_attn_materialized_fwd(q, k, v, out, probs, lse, workspace, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("out", out)], lse=lse, workspace=workspace)
    _check_probs(probs, B, Hq, T)
    _check(lib().rca_attn_materialized_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, T, Dh, _ptr(out), _ptr(probs),
                                           _ptr(lse), _dtype_code(q), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))


def rca_attn_materialized_bwd(q, k, v, probs, dout, dprobs, dq, dk, dv, workspace, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("dout", dout), ("dq", dq)],
                                   like_k=[("dk", dk), ("dv", dv)], workspace=workspace)
    _check_probs(probs, B, Hq, T)
    if dprobs is not None:
        _check_probs(dprobs, B, Hq, T, "dprobs")
    _check(lib().rca_attn_materialized_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(probs), _ptr(dout), _ptr(dprobs),
                                           _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, T, Dh, _dtype_code(q),
                                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))


def rca_causal_softmax(scores, lse, scale, stream=None):
    """In place on scores [N,T,T] float32 (any leading dims); lse [N,T] float32."""
    T = scores.shape[-1]
    N = scores.numel() // (T * T)
    _check(lib().rca_causal_softmax(_ptr(scores), _ptr(lse), N, T, float(scale), _stream(stream)))


def rca_causal_softmax_bwd(probs, grad, grad_extra, scale, stream=None):
    """In place on grad [N,T,T] float32; grad_extra may be None."""
    T = probs.shape[-1]
    N = probs.numel() // (T * T)
    _check(lib().rca_causal_softmax_bwd(_ptr(probs), _ptr(grad), _ptr(grad_extra), N, T, float(scale),
                                        _stream(stream)))


def rca_causal_softmax_bwd_tiled(probs, grad, grad_extra, tile, scale, stream=None):
    """As rca_causal_softmax_bwd, row i read and written only for columns
    j < min(T, tile * (i // tile + 1)); the rest of grad is left as it was."""
    T = probs.shape[-1]
    N = probs.numel() // (T * T)
    _check(lib().rca_causal_softmax_bwd_tiled(_ptr(probs), _ptr(grad), _ptr(grad_extra), N, T, int(tile),
                                              float(scale), _stream(stream)))


def _qkv_shape(qkv, Hq, Hkv):
    if qkv.dim() != 3 or qkv.shape[2] % (Hq + 2 * Hkv):
        raise ValueError("qkv must be [B, T, (Hq + 2*Hkv) * Dh]")
    B, T, W = qkv.shape
    return B, T, W // (Hq + 2 * Hkv)


def rca_attn_fwd_qkv(qkv, Hq, Hkv, out, lse, stream=None):
    B, T, Dh = _qkv_shape(qkv, Hq, Hkv)
    _check(lib().rca_attn_fwd_qkv(_ptr(qkv), B, T, Hq, Hkv, Dh, _ptr(out), _ptr(lse), _dtype_code(qkv),
                                  _stream(stream)))


def rca_attn_bwd_qkv(qkv, Hq, Hkv, out, lse, dout, dqkv, workspace, stream=None):
    B, T, Dh = _qkv_shape(qkv, Hq, Hkv)
    _check(lib().rca_attn_bwd_qkv(_ptr(qkv), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dqkv), B, T, Hq, Hkv, Dh,
                                  _dtype_code(qkv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def _check_lens(seq_lens, B):
    torch = _torch()
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be int32 [B]")


def rca_attn_varlen_workspace_size(B, Hq, Hkv, T, Dh, dt) -> int:
    """dt: RCA_BF16 / RCA_F32_TF32, or a torch dtype."""
    if not isinstance(dt, int):
        torch = _torch()
        dt = RCA_BF16 if dt == torch.bfloat16 else RCA_F32_TF32
    return lib().rca_attn_varlen_workspace_size(B, Hq, Hkv, T, Dh, dt)


def rca_attn_fwd_varlen(q, k, v, seq_lens, out, lse, workspace, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("out", out)], lse=lse, workspace=workspace)
    _check_lens(seq_lens, B)
    _check(lib().rca_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, Hq, Hkv, T, Dh, _ptr(out),
                                     _ptr(lse), _dtype_code(q), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def rca_attn_bwd_varlen(q, k, v, out, lse, dout, seq_lens, dq, dk, dv, workspace, stream=None):
    B, Hq, Hkv, T, Dh = _attn_args(q, k, v, like_q=[("out", out), ("dout", dout), ("dq", dq)],
                                   like_k=[("dk", dk), ("dv", dv)], lse=lse, workspace=workspace)
    _check_lens(seq_lens, B)
    _check(lib().rca_attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(seq_lens),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, T, Dh, _dtype_code(q),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def rca_selftest_device_timeout(stream=None):
    _check(lib().rca_selftest_device_timeout(_stream(stream)))


def rca_selftest_noalloc_timeout(stream=None):
    _check(lib().rca_selftest_noalloc_timeout(_stream(stream)))


def rca_stream_status(stream=None):
    _check(lib().rca_stream_status(_stream(stream)))
