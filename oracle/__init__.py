"""fp64 CPU oracle for kernelized linear attention (phi = elu + 1).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``linear_attention_02_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``la_oracle.c`` (plain C, fp64, one routine per form
the pages give); this module compiles it with gcc and marshals numpy/torch
arrays into contiguous float64 buffers.  See ``la_oracle.h`` for the citation
of each routine.

parity pins: every routine is pinned by ``tests/test_oracle_pins.py`` against
hand-derived values, closed forms, library routines and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liblaoracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile la_oracle.c into oracle/lib/liblaoracle.so (host gcc, no -march)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    hdr = os.path.join(_HERE, "la_oracle.h")
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.lao_phi.restype = ctypes.c_double
    lib.lao_phi.argtypes = [ctypes.c_double]
    lib.lao_dphi.restype = ctypes.c_double
    lib.lao_dphi.argtypes = [ctypes.c_double]
    lib.lao_default_threads.restype = I
    lib.lao_default_threads.argtypes = []
    lib.lao_causal_forward_quadratic.argtypes = [I, I, I, I, P, P, P, P]
    lib.lao_causal_forward_recurrent.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, I]
    lib.lao_noncausal_forward_quadratic.argtypes = [I, I, I, I, P, P, P, P]
    lib.lao_noncausal_forward_assoc.argtypes = [I, I, I, I, P, P, P, P, P, P, I]
    lib.lao_causal_backward_cumsum.argtypes = [I, I, I, I, P, P, P, P, P, P, P, I]
    lib.lao_causal_backward_quadratic.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
    lib.lao_decode_step.argtypes = [I, I, I, P, P, P, P, P, P]
    lib.lao_noncausal_backward_assoc.argtypes = [I, I, I, I, P, P, P, P, P, P, P, I]
    lib.lao_noncausal_backward_quadratic.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
    lib.lao_softmax_decode_step.argtypes = [I, I, I, I, P, P, P, P, P, P]
    lib.lao_retention_forward_recurrent.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P]
    lib.lao_retention_forward_quadratic.argtypes = [I, I, I, I, I, P, P, P, P, P, P]
    lib.lao_retention_decode_step.argtypes = [I, I, I, P, P, P, P, P, P]
    lib.lao_poly_forward_quadratic.argtypes = [I, I, I, I, P, P, P, P, I]
    lib.lao_poly_forward_state.argtypes = [I, I, I, I, P, P, P, P, I]
    for f in ("lao_causal_forward_quadratic", "lao_causal_forward_recurrent",
              "lao_noncausal_forward_quadratic", "lao_noncausal_forward_assoc",
              "lao_causal_backward_cumsum", "lao_causal_backward_quadratic", "lao_decode_step",
              "lao_noncausal_backward_assoc", "lao_noncausal_backward_quadratic",
              "lao_softmax_decode_step", "lao_retention_forward_recurrent",
              "lao_retention_forward_quadratic", "lao_retention_decode_step",
              "lao_poly_forward_quadratic", "lao_poly_forward_state"):
        getattr(lib, f).restype = None
    _lib = lib
    return lib


def _f64(x) -> np.ndarray:
    """Contiguous float64 copy of a numpy array or (CPU) torch tensor."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _heads(x, tail):
    """Shape [..., N, tail] -> (leading shape, nh, N)."""
    lead = x.shape[:-2]
    nh = int(np.prod(lead)) if len(lead) else 1
    return lead, nh, x.shape[-2]


def phi(x: float) -> float:
    return _load().lao_phi(float(x))


def dphi(x: float) -> float:
    return _load().lao_dphi(float(x))


def default_threads() -> int:
    return int(_load().lao_default_threads())


def causal_forward_quadratic(Q, K, V) -> np.ndarray:
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    O = np.empty(lead + (N, M))
    _load().lao_causal_forward_quadratic(nh, N, D, M, _p(Q), _p(K), _p(V), _p(O))
    return O


def causal_forward_recurrent(Q, K, V, S0=None, Z0=None, nthreads: int = 0, return_den=False):
    """Returns (O, S_N, Z_N), plus the per-token denominator phi(Q_t).Z_t
    (shape [..., N]) with return_den."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    S0 = None if S0 is None else _f64(S0)
    Z0 = None if Z0 is None else _f64(Z0)
    O = np.empty(lead + (N, M))
    S = np.empty(lead + (D, M))
    Z = np.empty(lead + (D,))
    den = np.empty(lead + (N,)) if return_den else None
    _load().lao_causal_forward_recurrent(nh, N, D, M, _p(Q), _p(K), _p(V), _p(S0), _p(Z0),
                                         _p(O), _p(S), _p(Z), _p(den), int(nthreads))
    return (O, S, Z, den) if return_den else (O, S, Z)


def noncausal_forward_quadratic(Q, K, V) -> np.ndarray:
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    O = np.empty(lead + (N, M))
    _load().lao_noncausal_forward_quadratic(nh, N, D, M, _p(Q), _p(K), _p(V), _p(O))
    return O


def noncausal_forward_assoc(Q, K, V, nthreads: int = 0):
    """Returns (O, S, Z)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    O = np.empty(lead + (N, M))
    S = np.empty(lead + (D, M))
    Z = np.empty(lead + (D,))
    _load().lao_noncausal_forward_assoc(nh, N, D, M, _p(Q), _p(K), _p(V), _p(O), _p(S), _p(Z),
                                        int(nthreads))
    return O, S, Z


def causal_backward_cumsum(Q, K, V, G, nthreads: int = 0):
    """Returns (dQ, dK, dV) of L = sum(G * O)."""
    Q, K, V, G = _f64(Q), _f64(K), _f64(V), _f64(G)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    _load().lao_causal_backward_cumsum(nh, N, D, M, _p(Q), _p(K), _p(V), _p(G), _p(dQ), _p(dK),
                                       _p(dV), int(nthreads))
    return dQ, dK, dV


def causal_backward_quadratic(Q, K, V, G):
    Q, K, V, G = _f64(Q), _f64(K), _f64(V), _f64(G)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    _load().lao_causal_backward_quadratic(nh, N, D, M, _p(Q), _p(K), _p(V), _p(G), _p(dQ), _p(dK),
                                          _p(dV))
    return dQ, dK, dV


def noncausal_backward_assoc(Q, K, V, G, nthreads: int = 0):
    """Returns (dQ, dK, dV) of L = sum(G * O) for the non-causal output."""
    Q, K, V, G = _f64(Q), _f64(K), _f64(V), _f64(G)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    _load().lao_noncausal_backward_assoc(nh, N, D, M, _p(Q), _p(K), _p(V), _p(G), _p(dQ), _p(dK),
                                         _p(dV), int(nthreads))
    return dQ, dK, dV


def noncausal_backward_quadratic(Q, K, V, G):
    Q, K, V, G = _f64(Q), _f64(K), _f64(V), _f64(G)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    _load().lao_noncausal_backward_quadratic(nh, N, D, M, _p(Q), _p(K), _p(V), _p(G), _p(dQ),
                                             _p(dK), _p(dV))
    return dQ, dK, dV


def decode_step(q, k, v, S, Z):
    """One decode step; returns (out, S_new, Z_new) without touching the inputs."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = _f64(S).copy()
    Z = _f64(Z).copy()
    D, M = q.shape[-1], v.shape[-1]
    nh = int(np.prod(q.shape[:-1])) if q.ndim > 1 else 1
    out = np.empty(q.shape[:-1] + (M,))
    _load().lao_decode_step(nh, D, M, _p(q), _p(k), _p(v), _p(S), _p(Z), _p(out))
    return out, S, Z


def softmax_decode_step(q, k, v, Kc, Vc):
    """Softmax KV-cache decode: out [..., M] for q, k [..., D], v [..., M] and
    caches Kc [..., T, D], Vc [..., T, M] of the T earlier positions."""
    q, k, v, Kc, Vc = _f64(q), _f64(k), _f64(v), _f64(Kc), _f64(Vc)
    D, M = q.shape[-1], v.shape[-1]
    T = Kc.shape[-2]
    nh = int(np.prod(q.shape[:-1])) if q.ndim > 1 else 1
    out = np.empty(q.shape[:-1] + (M,))
    _load().lao_softmax_decode_step(nh, T, D, M, _p(q), _p(k), _p(v), _p(Kc), _p(Vc), _p(out))
    return out


def _decays(Q, gamma_head, gates):
    gh = None if gamma_head is None else _f64(gamma_head).reshape(-1)
    gt = None if gates is None else _f64(gates)
    return gh, gt


def retention_forward_recurrent(Q, K, V, gamma_head=None, gates=None, S0=None):
    """Retention over [B, H, N, *] inputs; returns (O, S_N).  gamma_head: [H];
    gates: [B, H, N]; neither: decay 1."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, D = Q.shape
    M = V.shape[-1]
    gh, gt = _decays(Q, gamma_head, gates)
    S0 = None if S0 is None else _f64(S0)
    O = np.empty((B, H, N, M))
    S = np.empty((B, H, D, M))
    _load().lao_retention_forward_recurrent(B * H, H, N, D, M, _p(Q), _p(K), _p(V), _p(gh), _p(gt),
                                            _p(S0), _p(O), _p(S))
    return O, S


def retention_forward_quadratic(Q, K, V, gamma_head=None, gates=None):
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, D = Q.shape
    M = V.shape[-1]
    gh, gt = _decays(Q, gamma_head, gates)
    O = np.empty((B, H, N, M))
    _load().lao_retention_forward_quadratic(B * H, H, N, D, M, _p(Q), _p(K), _p(V), _p(gh), _p(gt),
                                            _p(O))
    return O


def retention_decode_step(q, k, v, gamma, S):
    """One step for every head: returns (out, S_new); gamma has one decay per head."""
    q, k, v, S = _f64(q), _f64(k), _f64(v), _f64(S).copy()
    D, M = q.shape[-1], v.shape[-1]
    nh = int(np.prod(q.shape[:-1]))
    g = np.ascontiguousarray(np.broadcast_to(np.asarray(gamma, dtype=np.float64), q.shape[:-1]))
    out = np.empty(q.shape[:-1] + (M,))
    _load().lao_retention_decode_step(nh, D, M, _p(q), _p(k), _p(v), _p(g), _p(S), _p(out))
    return out, S


def _poly(fn, Q, K, V, causal):
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, nh, N = _heads(Q, Q.shape[-1])
    D, M = Q.shape[-1], V.shape[-1]
    O = np.empty(lead + (N, M))
    fn(nh, N, D, M, _p(Q), _p(K), _p(V), _p(O), 1 if causal else 0)
    return O


def poly_forward_quadratic(Q, K, V, causal=True):
    """Attention with similarity (Q_i . K_j)^2, written out directly."""
    return _poly(_load().lao_poly_forward_quadratic, Q, K, V, causal)


def poly_forward_state(Q, K, V, causal=True):
    """The same through the explicit degree-2 feature map (C = D^2 state)."""
    return _poly(_load().lao_poly_forward_state, Q, K, V, causal)
