"""Python calls with the C ABI's names, on torch CUDA tensors.

Argument marshalling only: every step of the path runs in libhypic's CUDA
kernels.  Outputs are allocated with torch on the inputs' device; calls are
enqueued on torch's current stream.  See ``include/hypic.h`` for layouts.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib as L

_DT = {torch.float32: "f32", torch.bfloat16: "bf16"}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t, name, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def t_size(family: str, d: int) -> int:
    return 1 if family in ("scalar_const", "scalar") else (d if family == "diag" else d * d)


def _t_shape(family, lead, d):
    if family in ("scalar_const", "scalar"):
        return (*lead,)
    if family == "diag":
        return (*lead, d)
    return (*lead, d, d)


def _in_dtype(k):
    try:
        return _DT[k.dtype]
    except KeyError:
        raise ValueError(f"inputs must be float32 or bfloat16, got {k.dtype}") from None


def _gates(family, alpha, beta):
    alpha = _cuda(alpha, "alpha", torch.float32, allow_none=family == "delta")
    beta = _cuda(beta, "beta", torch.float32, allow_none=family not in ("delta", "gated_delta", "kda"))
    return alpha, beta


def segment_build(k, v, alpha=None, beta=None, q=None, family="gated_delta", want_o=False, stream=None):
    """(T_C, S_{C|0}[, o]) of one segment body: k, v, q [len, H, d]."""
    lib = L.load()
    _cuda(k, "k"), _cuda(v, "v", k.dtype)
    n, H, d = k.shape
    alpha, beta = _gates(family, alpha, beta)
    if want_o:
        _cuda(q, "q", k.dtype)
    sh = L.shape(H, d, family, _in_dtype(k))
    T = torch.empty((H, t_size(family, d)), device=k.device, dtype=torch.float32)
    S = torch.empty((H, d, d), device=k.device, dtype=torch.float32)
    o = torch.empty((n, H, d), device=k.device, dtype=torch.float32) if want_o else None
    query = lib.hypic_build_workspace_bytes_outputs if want_o else lib.hypic_build_workspace_bytes
    ws_bytes = query(ctypes.byref(sh), 1, n)
    ws = torch.empty(ws_bytes, device=k.device, dtype=torch.uint8) if ws_bytes else None
    st = lib.hypic_segment_build(ctypes.byref(sh), _p(k), _p(v), _p(q if want_o else None), _p(alpha), _p(beta), n,
                                 _p(T), _p(S), _p(o), _p(ws), ws_bytes, _stream(stream))
    L.check(st, "hypic_segment_build")
    T = T.view(_t_shape(family, (H,), d))
    return (T, S, o) if want_o else (T, S)


def build_workspace_bytes(H, d, n_seg, max_len, family="gated_delta", in_dtype="bf16", want_o=False) -> int:
    """Preferred workspace of a batched build (0 when the shape needs none)."""
    sh = L.shape(H, d, family, in_dtype)
    lib = L.load()
    query = lib.hypic_build_workspace_bytes_outputs if want_o else lib.hypic_build_workspace_bytes
    return int(query(ctypes.byref(sh), n_seg, max_len))


def segment_build_batched(k, v, bounds, alpha=None, beta=None, q=None, family="gated_delta", max_len=None,
                          want_o=False, out=None, ws=None, o_out=None, stream=None):
    """Pairs of n_seg bodies [begin, end) = bounds[i] (int64 [n_seg, 2] on the device) of one token axis."""
    lib = L.load()
    _cuda(k, "k"), _cuda(v, "v", k.dtype)
    _cuda(bounds, "bounds", torch.int64)
    n_tok, H, d = k.shape
    n_seg = bounds.shape[0]
    alpha, beta = _gates(family, alpha, beta)
    if want_o:
        _cuda(q, "q", k.dtype)
    if max_len is None:
        max_len = int((bounds[:, 1] - bounds[:, 0]).max().item()) if n_seg else 0
    sh = L.shape(H, d, family, _in_dtype(k))
    if out is None:
        T = torch.empty((n_seg, H, t_size(family, d)), device=k.device, dtype=torch.float32)
        S = torch.empty((n_seg, H, d, d), device=k.device, dtype=torch.float32)
    else:
        T, S = out
        _cuda(T, "T_out", torch.float32), _cuda(S, "S_out", torch.float32)
    if want_o and o_out is not None:
        o = _cuda(o_out, "o_out", torch.float32)
    else:
        o = torch.zeros((n_tok, H, d), device=k.device, dtype=torch.float32) if want_o else None
    if ws is None:
        query = lib.hypic_build_workspace_bytes_outputs if want_o else lib.hypic_build_workspace_bytes
        ws_bytes = query(ctypes.byref(sh), n_seg, max_len)
        ws = torch.empty(ws_bytes, device=k.device, dtype=torch.uint8) if ws_bytes else None
    else:
        _cuda(ws, "ws", torch.uint8)
        ws_bytes = ws.numel()
    st = lib.hypic_segment_build_batched(ctypes.byref(sh), n_seg, _p(bounds), max_len, n_tok, _p(k), _p(v),
                                         _p(q if want_o else None), _p(alpha), _p(beta), _p(T), _p(S), _p(o),
                                         _p(ws), ws_bytes, _stream(stream))
    L.check(st, "hypic_segment_build_batched")
    T = T.view(_t_shape(family, (n_seg, H), d))
    return (T, S, o) if want_o else (T, S)


def _host(t, name, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor (pinned for asynchronous copies)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def segment_build_batched_host(k, v, bounds, alpha=None, beta=None, family="gated_delta", max_len=None,
                               dev=None, out=None, ws=None, stream=None, copy_stream=None, ready_event=None,
                               device="cuda"):
    """The batched build from host tensors (pinned memory: the copies overlap the build).

    k, v [n_tok, H, d], alpha/beta and bounds (int64 [n_seg, 2]) live on the host.  ``dev`` is a
    tuple of device buffers (k, v, alpha, beta, bounds) of the same shapes (allocated when None);
    the copies run on ``copy_stream`` (a new stream when None) while earlier segment groups build
    on ``stream``.  ``ready_event`` (a torch.cuda.Event) marks when nothing reads the ``dev`` buffers
    any more; without it the copies wait for all work already on ``stream``.  Returns (T, S) on the
    device, ready on ``stream``."""
    lib = L.load()
    _host(k, "k"), _host(v, "v", k.dtype), _host(bounds, "bounds", torch.int64)
    n_tok, H, d = k.shape
    n_seg = bounds.shape[0]
    alpha = _host(alpha, "alpha", torch.float32, allow_none=family == "delta")
    beta = _host(beta, "beta", torch.float32, allow_none=family not in ("delta", "gated_delta", "kda"))
    if max_len is None:
        max_len = int((bounds[:, 1] - bounds[:, 0]).max().item()) if n_seg else 0
    if dev is None:
        dev = tuple(None if t is None else torch.empty(t.shape, dtype=t.dtype, device=device)
                    for t in (k, v, alpha, beta, bounds))
    k_d, v_d, a_d, b_d, bn_d = dev
    _cuda(k_d, "k_dev", k.dtype), _cuda(v_d, "v_dev", k.dtype), _cuda(bn_d, "bounds_dev", torch.int64)
    if alpha is not None:
        _cuda(a_d, "alpha_dev", torch.float32)
    if beta is not None:
        _cuda(b_d, "beta_dev", torch.float32)
    sh = L.shape(H, d, family, _in_dtype(k))
    if out is None:
        T = torch.empty((n_seg, H, t_size(family, d)), device=k_d.device, dtype=torch.float32)
        S = torch.empty((n_seg, H, d, d), device=k_d.device, dtype=torch.float32)
    else:
        T, S = out
        _cuda(T, "T_out", torch.float32), _cuda(S, "S_out", torch.float32)
    if ws is None:
        ws_bytes = lib.hypic_build_workspace_bytes(ctypes.byref(sh), n_seg, max_len)
        ws = torch.empty(ws_bytes, device=k_d.device, dtype=torch.uint8) if ws_bytes else None
    else:
        _cuda(ws, "ws", torch.uint8)
        ws_bytes = ws.numel()
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=k_d.device)
    st = lib.hypic_segment_build_batched_host(ctypes.byref(sh), n_seg, ctypes.c_void_p(bounds.data_ptr()), max_len,
                                              n_tok, ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                              None if alpha is None else ctypes.c_void_p(alpha.data_ptr()),
                                              None if beta is None else ctypes.c_void_p(beta.data_ptr()),
                                              _p(k_d), _p(v_d), _p(a_d if alpha is not None else None),
                                              _p(b_d if beta is not None else None), _p(bn_d), _p(T), _p(S), _p(ws),
                                              ws_bytes, _stream(stream), _stream(copy_stream),
                                              None if ready_event is None else ctypes.c_void_p(ready_event.cuda_event))
    L.check(st, "hypic_segment_build_batched_host")
    return T.view(_t_shape(family, (n_seg, H), d)), S


def _pool_dtype(pool_T, pool_S):
    """fp32 pools, or bf16 pools (16-bit pair storage, see pairs_to_bf16); both the same."""
    dt = pool_S.dtype if isinstance(pool_S, torch.Tensor) else None
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("pool_S must be a float32 or bfloat16 CUDA tensor")
    _cuda(pool_S, "pool_S", dt), _cuda(pool_T, "pool_T", dt)
    return dt == torch.bfloat16


def pairs_to_bf16(T, S, family="gated_delta", stream=None):
    """Round fp32 pairs T [n, H, ...], S [n, H, d, d] to bf16 storage (nearest even)."""
    lib = L.load()
    _cuda(T, "T", torch.float32), _cuda(S, "S", torch.float32)
    n, H, d, _ = S.shape
    T_lp = torch.empty(T.shape, device=S.device, dtype=torch.bfloat16)
    S_lp = torch.empty(S.shape, device=S.device, dtype=torch.bfloat16)
    sh = L.shape(H, d, family, "f32")
    st = lib.hypic_pairs_to_bf16(ctypes.byref(sh), n, _p(T), _p(S), _p(T_lp), _p(S_lp), _stream(stream))
    L.check(st, "hypic_pairs_to_bf16")
    return T_lp, S_lp


def compose(pool_T, pool_S, idx, S_init=None, family="gated_delta", out=None, stream=None):
    """S_out [B, H, d, d]: each request b composes pool entries idx[b, 0..n-1] in order.

    The pools are fp32, or bf16 as written by pairs_to_bf16 (hypic_compose_bf16)."""
    lib = L.load()
    lp = _pool_dtype(pool_T, pool_S)
    _cuda(idx, "idx", torch.int32)
    P, H, d, _ = pool_S.shape
    B, n = idx.shape
    if S_init is not None:
        _cuda(S_init, "S_init", torch.float32)
    S_out = out if out is not None else torch.empty((B, H, d, d), device=pool_S.device, dtype=torch.float32)
    sh = L.shape(H, d, family, "f32")
    fn, name = (lib.hypic_compose_bf16, "hypic_compose_bf16") if lp else (lib.hypic_compose, "hypic_compose")
    st = fn(ctypes.byref(sh), B, n, _p(idx), P, _p(pool_T), _p(pool_S), _p(S_init), _p(S_out), _stream(stream))
    L.check(st, name)
    return S_out


def affine_scan(T, S, family="gated_delta", stream=None, two_level=True):
    """Inclusive prefix scan of n pairs: T [n, H, ...], S [n, H, d, d].  two_level=False passes no
    workspace, so every head's scan runs as one sequential chain."""
    lib = L.load()
    _cuda(T, "T", torch.float32), _cuda(S, "S", torch.float32)
    n, H, d, _ = S.shape
    sh = L.shape(H, d, family, "f32")
    Tp = torch.empty_like(T)
    Sp = torch.empty_like(S)
    ws_bytes = lib.hypic_scan_workspace_bytes(ctypes.byref(sh), n) if two_level else 0
    ws = torch.empty(ws_bytes, device=S.device, dtype=torch.uint8) if ws_bytes else None
    st = lib.hypic_affine_scan(ctypes.byref(sh), n, _p(T), _p(S), _p(Tp), _p(Sp), _p(ws), ws_bytes,
                               _stream(stream))
    L.check(st, "hypic_affine_scan")
    return Tp, Sp


def seam_advance(S, k, v, alpha=None, beta=None, q=None, family="gated_delta", want_o=True, stream=None):
    """Advance S [B, H, d, d] in place through seam tokens k, v, q [B, w, H, d]; returns o [B, w, H, d]."""
    lib = L.load()
    _cuda(S, "S", torch.float32), _cuda(k, "k"), _cuda(v, "v", k.dtype)
    B, w, H, d = k.shape
    alpha, beta = _gates(family, alpha, beta)
    if want_o:
        _cuda(q, "q", k.dtype)
    o = torch.empty((B, w, H, d), device=k.device, dtype=torch.float32) if want_o else None
    sh = L.shape(H, d, family, _in_dtype(k))
    st = lib.hypic_seam_advance(ctypes.byref(sh), B, _p(S), _p(q if want_o else None), _p(k), _p(v), _p(alpha),
                                _p(beta), w, _p(o), _stream(stream))
    L.check(st, "hypic_seam_advance")
    return o


def assemble(pool_T, pool_S, idx, seam_k, seam_v, seam_alpha=None, seam_beta=None, seam_q=None,
             S_init=None, family="gated_delta", want_o=True, out=None, o_out=None, stream=None):
    """Fused seam advance + compose.  Seam tokens [B, n-1, w, H, d]; returns (S_out, o [B, n-1, w, H, d]).

    The pools are fp32, or bf16 as written by pairs_to_bf16 (hypic_assemble_bf16)."""
    lib = L.load()
    lp = _pool_dtype(pool_T, pool_S)
    _cuda(idx, "idx", torch.int32)
    P, H, d, _ = pool_S.shape
    B, n = idx.shape
    w = seam_k.shape[2] if seam_k is not None and seam_k.dim() == 5 else 0
    if w > 0 and n > 1:
        _cuda(seam_k, "seam_k"), _cuda(seam_v, "seam_v", seam_k.dtype)
        seam_alpha, seam_beta = _gates(family, seam_alpha, seam_beta)
        if want_o:
            _cuda(seam_q, "seam_q", seam_k.dtype)
        in_dtype = _in_dtype(seam_k)
    else:
        in_dtype = "f32"
    if S_init is not None:
        _cuda(S_init, "S_init", torch.float32)
    S_out = out if out is not None else torch.empty((B, H, d, d), device=pool_S.device, dtype=torch.float32)
    o = None
    if want_o and w > 0 and n > 1:
        o = o_out if o_out is not None else torch.empty((B, n - 1, w, H, d), device=pool_S.device,
                                                        dtype=torch.float32)
    sh = L.shape(H, d, family, in_dtype)
    fn, name = (lib.hypic_assemble_bf16, "hypic_assemble_bf16") if lp else (lib.hypic_assemble, "hypic_assemble")
    st = fn(ctypes.byref(sh), B, n, w, _p(idx), P, _p(pool_T), _p(pool_S), _p(seam_q if o is not None else None),
            _p(seam_k), _p(seam_v), _p(seam_alpha), _p(seam_beta), _p(S_init), _p(S_out), _p(o), _stream(stream))
    L.check(st, name)
    return S_out, o


# ---- boundary patches (HYPIC notes, Method 6; paper Eqs. (7), (8)) ------------------------

_ACT = {"identity": 0, "silu": 1}


def _dt(t):
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise ValueError(f"expected float32 or bfloat16, got {t.dtype}")


def rope_shift(K, delta, rot_dim=None, base=10000.0, out=None, stream=None):
    """K_b = R(delta) K_a on the last axis of K [..., d] (rotate-half pairs, rot_dim dims rotated)."""
    lib = L.load()
    _cuda(K, "K")
    d = K.shape[-1]
    rows = K.numel() // d if d else 0
    out = out if out is not None else torch.empty_like(K)
    _cuda(out, "out", K.dtype)
    st = lib.hypic_rope_shift(rows, d, rot_dim or d, float(base), int(delta), _dt(K), _p(K), _p(out), _stream(stream))
    L.check(st, "hypic_rope_shift")
    return out


def state_rerotate(S, delta, rot_dim=None, base=10000.0, family="scalar", stream=None):
    """S_{C|b} = R(delta) S_{C|a} in place on the rows of S [n, H, d_k, d_v] (scalar families only)."""
    lib = L.load()
    _cuda(S, "S", torch.float32)
    n, H, dk, dv = S.shape
    sh = L.shape(H, dk, family, "f32")
    sh.d_v = dv
    st = lib.hypic_state_rerotate(ctypes.byref(sh), n, _p(S), rot_dim or dk, float(base), int(delta), _stream(stream))
    L.check(st, "hypic_state_rerotate")
    return S


def conv_tail(x, bounds, k, stream=None):
    """Last k - 1 inputs of each body [begin, end) = bounds[s] of x [n_tokens, C] -> [n_seg, k-1, C]."""
    lib = L.load()
    _cuda(x, "x"), _cuda(bounds, "bounds", torch.int64)
    n_tokens, C = x.shape
    n_seg = bounds.shape[0]
    tail = torch.zeros((n_seg, max(k - 1, 0), C), device=x.device, dtype=x.dtype)
    st = lib.hypic_conv_tail(C, k, n_seg, _p(bounds), n_tokens, _dt(x), _p(x), _p(tail), _stream(stream))
    L.check(st, "hypic_conv_tail")
    return tail


def conv_seam(x_seam, tail, weight, bias=None, act="identity", stream=None):
    """Causal conv outputs of the first w tokens of B segments: x_seam [B, w, C], tail [B, k-1, C]."""
    lib = L.load()
    _cuda(x_seam, "x_seam"), _cuda(weight, "weight", torch.float32)
    B, w, C = x_seam.shape
    k = weight.shape[1]
    if k > 1:
        _cuda(tail, "tail", x_seam.dtype)
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    y = torch.empty((B, w, C), device=x_seam.device, dtype=torch.float32)
    st = lib.hypic_conv_seam(B, w, C, k, _dt(x_seam), _p(x_seam), _p(tail if k > 1 else None), _p(weight), _p(bias),
                             _ACT[act], _p(y), _stream(stream))
    L.check(st, "hypic_conv_seam")
    return y


def stream_status(stream=None) -> int:
    """Wait for the stream; return and clear the device status word (0 = no error recorded)."""
    return int(L.load().hypic_stream_status(_stream(stream)))
