"""GB300 (sm_103a) kernelized linear attention, phi(x) = elu(x) + 1.

Thin Python binding over the C ABI of include/linattn.h.  The functions carry
the C names and only marshal arguments: torch supplies device memory and the
current CUDA stream; every step of the computation runs in liblinattn.so.

    la_forward_causal(Q, K, V, ...)      V'_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i, j <= i
    la_backward_causal(Q, K, V, dOut, ...)
    la_forward_noncausal(Q, K, V, ...)   phi(Q)(phi(K)^T V) / phi(Q) sum phi(K)
    la_decode_step(q, k, v, S, Z, ...)   S += phi(k)v^T, Z += phi(k); read with q

Shapes: Q, K [B,H,N,D]; V [B,H,N,M]; S [B,H,D,M] fp32; Z [B,H,D] fp32.
"""
from __future__ import annotations

import torch

from . import _native

_lib = _native.lib

_DT = {torch.float32: _native.LA_DTYPE_F32, torch.bfloat16: _native.LA_DTYPE_BF16}


class LinAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_lib.la_status_string(status).decode()}: {msg}")
        self.status = status


def _check(status: int) -> None:
    if status != _native.LA_OK:
        raise LinAttnError(status, (_lib.la_last_error_message() or b"").decode())


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _dims(Q, V):
    if Q.dim() != 4 or V.dim() != 4:
        raise ValueError("Q/K must be [B,H,N,D] and V [B,H,N,M]")
    B, H, N, D = Q.shape
    if tuple(V.shape[:3]) != (B, H, N):
        raise ValueError(f"V shape {tuple(V.shape)} does not match Q {tuple(Q.shape)}")
    return B, H, N, D, V.shape[3]


def _dtype(t):
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")
    return _DT[t.dtype]


def la_causal_ckpt_floats(B, H, N, D, M):
    """fp32 words of the optional state checkpoints (la_forward_causal(ckpt=...))."""
    return int(_lib.la_causal_ckpt_floats(B, H, N, D, M))


def la_forward_causal(Q, K, V, out=None, S_init=None, Z_init=None, return_state=False,
                      den=None, ckpt=None, stream=None):
    """Causal forward.  Returns Out, or (Out, S_final, Z_final) with return_state.

    den: optional fp32 [B, H, N] tensor that receives the normaliser
    phi(Q_i).Z_i of every token, to hand to la_backward_causal(Den=...).
    ckpt: optional fp32 tensor of la_causal_ckpt_floats(B, H, N, D, M) elements
    that receives state checkpoints, to hand to la_backward_causal(Ckpt=...)."""
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, Q.dtype, dev)
    if K.shape != Q.shape:
        raise ValueError("K must have the shape of Q")
    if out is None:
        out = torch.empty((B, H, N, M), dtype=Q.dtype, device=dev)
    _need(out, "out", Q.dtype, dev)
    if (S_init is None) != (Z_init is None):
        raise ValueError("give both S_init and Z_init, or neither")
    if S_init is not None:
        _need(S_init, "S_init", torch.float32, dev)
        _need(Z_init, "Z_init", torch.float32, dev)
    if den is not None:
        _need(den, "den", torch.float32, dev)
        if tuple(den.shape) != (B, H, N):
            raise ValueError(f"den must be [B, H, N] = {(B, H, N)}, got {tuple(den.shape)}")
    _check_ckpt(ckpt, "ckpt", B, H, N, D, M, dev)
    S_f = Z_f = None
    if return_state:
        S_f = torch.empty((B, H, D, M), dtype=torch.float32, device=dev)
        Z_f = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.la_forward_causal(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, N, D, M,
                                      _dtype(Q), _ptr(S_init), _ptr(Z_init), _ptr(S_f), _ptr(Z_f),
                                      _ptr(den), _ptr(ckpt), _stream_handle(stream)))
    return (out, S_f, Z_f) if return_state else out


def _check_ckpt(c, name, B, H, N, D, M, dev):
    if c is None:
        return
    _need(c, name, torch.float32, dev)
    if c.numel() != la_causal_ckpt_floats(B, H, N, D, M):
        raise ValueError(f"{name} must hold la_causal_ckpt_floats(...) = "
                         f"{la_causal_ckpt_floats(B, H, N, D, M)} floats, got {c.numel()}")


def la_backward_causal(Q, K, V, dOut, Out=None, dQ=None, dK=None, dV=None, Den=None,
                       Ckpt=None, stream=None):
    """Causal backward; returns (dQ, dK, dV).  Out (the forward output), Den
    (its normaliser, fp32 [B, H, N]) and Ckpt (its state checkpoints) are optional."""
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (dOut, "dOut")):
        _need(t, n, Q.dtype, dev)
    if Out is not None:
        _need(Out, "Out", Q.dtype, dev)
    if Den is not None:
        _need(Den, "Den", torch.float32, dev)
        if tuple(Den.shape) != (B, H, N):
            raise ValueError(f"Den must be [B, H, N] = {(B, H, N)}, got {tuple(Den.shape)}")
    _check_ckpt(Ckpt, "Ckpt", B, H, N, D, M, dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for t, n in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
        _need(t, n, Q.dtype, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_backward_causal(_ptr(Q), _ptr(K), _ptr(V), _ptr(Out), _ptr(dOut), _ptr(dQ),
                                       _ptr(dK), _ptr(dV), B, H, N, D, M, _dtype(Q), _ptr(Den),
                                       _ptr(Ckpt), _stream_handle(stream)))
    return dQ, dK, dV


def la_forward_noncausal(Q, K, V, out=None, stream=None):
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, Q.dtype, dev)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=Q.dtype, device=dev)
    _need(out, "out", Q.dtype, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_forward_noncausal(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, N, D, M,
                                         _dtype(Q), _stream_handle(stream)))
    return out


def la_backward_noncausal(Q, K, V, dOut, Out=None, dQ=None, dK=None, dV=None, stream=None):
    """Backward of la_forward_noncausal; returns (dQ, dK, dV).  Out is optional."""
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (dOut, "dOut")):
        _need(t, n, Q.dtype, dev)
    if K.shape != Q.shape or dOut.shape != V.shape:
        raise ValueError("K must have the shape of Q and dOut the shape of V")
    if Out is not None:
        _need(Out, "Out", Q.dtype, dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for t, n in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
        _need(t, n, Q.dtype, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_backward_noncausal(_ptr(Q), _ptr(K), _ptr(V), _ptr(Out), _ptr(dOut), _ptr(dQ),
                                          _ptr(dK), _ptr(dV), B, H, N, D, M, _dtype(Q),
                                          _stream_handle(stream)))
    return dQ, dK, dV


def la_forward_noncausal_noalloc(Q, K, V, out=None, stream=None):
    """la_forward_noncausal for callers that may not allocate device memory.

    The library side allocates nothing (its scratch is a fixed 16 MiB device
    array); pass `out` to keep this Python wrapper from allocating the output.
    Calls that overlap on the GPU share that array and must be serialised.
    """
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, Q.dtype, dev)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=Q.dtype, device=dev)
    _need(out, "out", Q.dtype, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_forward_noncausal_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, N, D,
                                                 M, _dtype(Q), _stream_handle(stream)))
    return out


def la_decode_step(q, k, v, S, Z, out=None, stream=None):
    """One decode step; updates S, Z in place and returns out [B,H,M] fp32."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q/k must be [B,H,D] and v [B,H,M]")
    B, H, D = q.shape
    M = v.shape[2]
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(S, "S", torch.float32, dev)
    _need(Z, "Z", torch.float32, dev)
    if tuple(S.shape) != (B, H, D, M) or tuple(Z.shape) != (B, H, D):
        raise ValueError("S must be [B,H,D,M] and Z [B,H,D]")
    if out is None:
        out = torch.empty((B, H, M), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(Z), _ptr(out), B, H, D,
                                   M, _dtype(q), _stream_handle(stream)))
    return out


def la_workspace_bytes(op, B, H, N, D, M, dtype, saved=0, num_sms=0):
    """Scratch bytes one call of entry point `op` takes from the library pool.

    dtype: torch.float32 or torch.bfloat16.  saved: OR of LA_SAVED_OUT,
    LA_SAVED_DEN, LA_SAVED_CKPT (la_backward_causal's optional inputs).
    num_sms <= 0 asks the current device for its SM count."""
    if dtype not in _DT:
        raise ValueError(f"unsupported dtype {dtype}")
    n = _lib.la_workspace_bytes(op.encode(), B, H, N, D, M, _DT[dtype], int(saved), int(num_sms))
    if n == _native.SIZE_MAX:
        raise LinAttnError(_native.LA_ERR_INVALID_ARG, la_last_error_message())
    return int(n)


def la_scratch_peak_bytes(reset=False):
    """Peak bytes of the library's scratch pool held at once on the current device."""
    n = _lib.la_scratch_peak_bytes(1 if reset else 0)
    if n == _native.SIZE_MAX:
        raise LinAttnError(_native.LA_ERR_CUDA, la_last_error_message())
    return int(n)


LA_SAVED_OUT, LA_SAVED_DEN, LA_SAVED_CKPT = (_native.LA_SAVED_OUT, _native.LA_SAVED_DEN,
                                             _native.LA_SAVED_CKPT)


def la_forward_poly2(Q, K, V, causal=True, out=None, stream=None):
    """Attention with similarity (Q_i . K_j)^2 through its degree-2 feature map (D = 32)."""
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, Q.dtype, dev)
    if K.shape != Q.shape:
        raise ValueError("K must have the shape of Q")
    if out is None:
        out = torch.empty((B, H, N, M), dtype=Q.dtype, device=dev)
    _need(out, "out", Q.dtype, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_forward_poly2(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, N, D, M, _dtype(Q),
                                     1 if causal else 0, _stream_handle(stream)))
    return out


def _decay_args(gamma_head, gates, shape, dev, name):
    if gamma_head is not None and gates is not None:
        raise ValueError(f"give gamma_head or {name}, not both")
    if gamma_head is not None:
        _need(gamma_head, "gamma_head", torch.float32, dev)
        if tuple(gamma_head.shape) != (shape[1],):
            raise ValueError(f"gamma_head must be [H] = {(shape[1],)}")
    if gates is not None:
        _need(gates, name, torch.float32, dev)
        if tuple(gates.shape) != tuple(shape):
            raise ValueError(f"{name} must be {tuple(shape)}, got {tuple(gates.shape)}")


def la_forward_retention(Q, K, V, gamma_head=None, gates=None, out=None, S_init=None,
                         return_state=False, stream=None):
    """Linear attention with decay: S_t = gamma_t S_{t-1} + k_t v_t^T, Out_t = S_t^T q_t.

    gamma_head [H] (RetNet), gates [B,H,N] (gated retention) or neither (decay 1).
    Returns Out, or (Out, S_final) with return_state."""
    B, H, N, D, M = _dims(Q, V)
    dev = Q.device
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, Q.dtype, dev)
    if K.shape != Q.shape:
        raise ValueError("K must have the shape of Q")
    _decay_args(gamma_head, gates, (B, H, N), dev, "gates")
    if out is None:
        out = torch.empty((B, H, N, M), dtype=Q.dtype, device=dev)
    _need(out, "out", Q.dtype, dev)
    if S_init is not None:
        _need(S_init, "S_init", torch.float32, dev)
    S_f = torch.empty((B, H, D, M), dtype=torch.float32, device=dev) if return_state else None
    with torch.cuda.device(dev):
        _check(_lib.la_forward_retention(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, N, D, M,
                                         _dtype(Q), _ptr(gamma_head), _ptr(gates), _ptr(S_init),
                                         _ptr(S_f), _stream_handle(stream)))
    return (out, S_f) if return_state else out


def la_retention_decode_step(q, k, v, S, gamma_head=None, gate=None, out=None, stream=None):
    """One retention step: S = gamma S + k v^T (in place), returns out = S^T q [B,H,M] fp32."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q/k must be [B,H,D] and v [B,H,M]")
    B, H, D = q.shape
    M = v.shape[2]
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(S, "S", torch.float32, dev)
    if tuple(S.shape) != (B, H, D, M):
        raise ValueError("S must be [B,H,D,M]")
    _decay_args(gamma_head, gate, (B, H), dev, "gate")
    if out is None:
        out = torch.empty((B, H, M), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_retention_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma_head), _ptr(gate),
                                             _ptr(S), _ptr(out), B, H, D, M, _dtype(q),
                                             _stream_handle(stream)))
    return out


def la_softmax_decode_step(q, k, v, K_cache, V_cache, T, out=None, stream=None):
    """Softmax attention decode step with a KV cache (the comparator of la_decode_step).

    Writes k, v into row T of K_cache [B,H,T_max,D] / V_cache [B,H,T_max,M] and
    returns out [B,H,M] fp32 = softmax(q K^T / sqrt(D)) V over rows 0..T."""
    if q.dim() != 3 or v.dim() != 3 or K_cache.dim() != 4 or V_cache.dim() != 4:
        raise ValueError("q, k [B,H,D], v [B,H,M], caches [B,H,T_max,D] / [B,H,T_max,M]")
    B, H, D = q.shape
    M = v.shape[2]
    T_max = K_cache.shape[2]
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (K_cache, "K_cache"), (V_cache, "V_cache")):
        _need(t, n, q.dtype, dev)
    if tuple(K_cache.shape) != (B, H, T_max, D) or tuple(V_cache.shape) != (B, H, T_max, M):
        raise ValueError("cache shapes do not match q and v")
    if out is None:
        out = torch.empty((B, H, M), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    with torch.cuda.device(dev):
        _check(_lib.la_softmax_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(K_cache), _ptr(V_cache),
                                           int(T), T_max, _ptr(out), B, H, D, M, _dtype(q),
                                           _stream_handle(stream)))
    return out


def la_check_device_status(stream=None):
    _check(_lib.la_check_device_status(_stream_handle(stream)))


def la_selftest_expired_waits(stream=None):
    """Launch a block whose bounded device waits expire (tests the error-word path).

    The next la_check_device_status() raises LinAttnError with LA_ERR_TIMEOUT.
    """
    _check(_lib.la_selftest_expired_waits(_stream_handle(stream)))


def la_kernel_launch_count() -> int:
    return int(_lib.la_kernel_launch_count())


def la_status_string(status: int) -> str:
    return _lib.la_status_string(int(status)).decode()


def la_last_error_message() -> str:
    return (_lib.la_last_error_message() or b"").decode()
