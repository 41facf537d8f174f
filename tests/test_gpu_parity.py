"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Error measure, per output tensor: max|got - ref| / max|ref| over the compared
elements, where ref is the oracle evaluated in fp64 on the very inputs the GPU
saw (bf16 values upcast exactly).  Tolerances: 1e-4 for fp32 storage and 2e-2
for bf16 storage, with fp32 accumulation on the GPU in both cases.

Small cases cover every (dtype, D, M) family, several chunks and spans, ragged
tails, N = 1 and N = 0.  Full-size cases run the exact shapes and launch
configuration the bench times and compare sampled heads (the oracle computes
each head independently), plus bounds that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def _la():
    import linear_attention_02_gb300 as la
    return la


def rel_err(got, ref) -> float:
    got = np.asarray(got.float().cpu().numpy() if isinstance(got, torch.Tensor) else got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def _dev(x):
    return {k: v.cuda() for k, v in x.items()}


SMALL = [
    # (B, H, N, D, M)
    (1, 1, 256, 32, 32),
    (2, 3, 200, 64, 32),
    (1, 2, 517, 128, 64),
    (2, 2, 1000, 64, 64),
    (1, 2, 130, 32, 128),
    (1, 1, 1, 64, 64),
    (1, 3, 77, 128, 128),
    (3, 1, 2049, 64, 128),
]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL)
def test_causal_forward_small(dt, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, dt, seed=11 + N)
    g = _dev(x)
    den = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    O, S, Z = la.la_forward_causal(g["Q"], g["K"], g["V"], return_state=True, den=den)
    torch.cuda.synchronize()
    Ro, Rs, Rz, Rd = oracle.causal_forward_recurrent(x["Q"], x["K"], x["V"], return_den=True)
    assert rel_err(O, Ro) <= TOL[dt]
    assert rel_err(S, Rs) <= TOL[dt]
    assert rel_err(Z, Rz) <= TOL[dt]
    assert rel_err(den, Rd) <= TOL[dt]


# The tensor-core kernels cut the chunks of all heads (head-major) into equal
# ranges, one per resident CTA: a range can hold the tail of one head, whole
# heads and the start of another, or a piece in the middle of a head.
@pytest.mark.parametrize("shape", [
    (8, 64, 300, 64, 64),     # many short heads: ranges of several heads each, ragged tails
    (1, 2, 5000, 128, 128),   # few heads: one chunk per range, ragged last chunk
    (1, 1, 128, 64, 64),      # exactly one chunk
    (2, 3, 129, 64, 64),      # one full chunk and a single-token tail
    (1, 4, 4096, 64, 64),
    (2, 3, 8300, 64, 64),     # several chunks per range, ranges crossing heads, ragged last chunk
    (4, 16, 2048, 64, 64),    # four ranges per head: pieces inside heads, look-back over aggregates only
    (1, 1, 20000, 64, 64),    # 157 one-chunk ranges in one head: the look-back stops at published head states
])
def test_causal_forward_bf16_span_shapes(shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "bf16", seed=13 + N)
    g = _dev(x)
    den = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    O, S, Z = la.la_forward_causal(g["Q"], g["K"], g["V"], return_state=True, den=den)
    la.la_check_device_status()
    idx = list(range(min(B * H, 6)))
    hs = [x[n].reshape(B * H, N, -1)[idx] for n in ("Q", "K", "V")]
    Ro, Rs, Rz, Rd = oracle.causal_forward_recurrent(*hs, return_den=True)
    assert rel_err(O.reshape(B * H, N, M)[idx], Ro) <= TOL["bf16"]
    assert rel_err(S.reshape(B * H, D, M)[idx], Rs) <= TOL["bf16"]
    assert rel_err(Z.reshape(B * H, D)[idx], Rz) <= TOL["bf16"]
    assert rel_err(den.reshape(B * H, N)[idx], Rd) <= TOL["bf16"]


@pytest.mark.parametrize("shape", [(1, 2, 3000, 64, 64), (2, 3, 8300, 64, 64)])
def test_causal_forward_checkpoints(shape):
    # slot k holds the state (S, Z) after the first 1024 k tokens of each head
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "bf16", seed=29 + N)
    g = _dev(x)
    ck = torch.full((la.la_causal_ckpt_floats(B, H, N, D, M),), float("nan"), device="cuda")
    la.la_forward_causal(g["Q"], g["K"], g["V"], ckpt=ck)
    la.la_check_device_status()
    slots = -(-(-(-N // 128)) // 8)
    ck = ck.reshape(B * H, slots, D * M + D)
    assert bool(torch.isnan(ck[:, 0]).all())  # slot 0 (the zero state) is left alone
    heads = [x[n].reshape(B * H, N, -1)[:2] for n in ("Q", "K", "V")]
    for k in range(1, slots):
        _, Rs, Rz = oracle.causal_forward_recurrent(*(h[:, :1024 * k] for h in heads))
        got = ck[:2, k]
        assert rel_err(got[:, :D * M].reshape(2, D, M), Rs) <= TOL["bf16"]
        assert rel_err(got[:, D * M:], Rz) <= TOL["bf16"]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_causal_forward_carried_state_and_empty(dt):
    la = _la()
    B, H, N, D, M, cut = 2, 2, 700, 64, 64, 333
    x = synth.qkv(B, H, N, D, M, dt, seed=5)
    g = _dev(x)
    Oa, Sa, Za = la.la_forward_causal(g["Q"][:, :, :cut].contiguous(), g["K"][:, :, :cut].contiguous(),
                                      g["V"][:, :, :cut].contiguous(), return_state=True)
    Ob, Sb, Zb = la.la_forward_causal(g["Q"][:, :, cut:].contiguous(), g["K"][:, :, cut:].contiguous(),
                                      g["V"][:, :, cut:].contiguous(), S_init=Sa, Z_init=Za,
                                      return_state=True)
    # an empty piece passes the state through unchanged
    e = torch.empty((B, H, 0, D), dtype=g["Q"].dtype, device="cuda")
    ev = torch.empty((B, H, 0, M), dtype=g["Q"].dtype, device="cuda")
    _, Se, Ze = la.la_forward_causal(e, e, ev, S_init=Sb, Z_init=Zb, return_state=True)
    torch.cuda.synchronize()
    Ro, Rs, Rz = oracle.causal_forward_recurrent(x["Q"], x["K"], x["V"])
    assert rel_err(torch.cat([Oa, Ob], 2), Ro) <= TOL[dt]
    assert rel_err(Sb, Rs) <= TOL[dt] and rel_err(Zb, Rz) <= TOL[dt]
    assert torch.equal(Se, Sb) and torch.equal(Ze, Zb)


def _saved(la, g, saved):
    """The forward's outputs handed to the backward: none, Out, Out and den, or Out, den
    and the state checkpoints."""
    if saved == "none":
        return None, None, None
    B, H, N, D = g["Q"].shape
    M = g["V"].shape[3]
    den = torch.empty((B, H, N), dtype=torch.float32, device="cuda") if "den" in saved else None
    ck = (torch.empty(la.la_causal_ckpt_floats(B, H, N, D, M), dtype=torch.float32, device="cuda")
          if "ckpt" in saved else None)
    return la.la_forward_causal(g["Q"], g["K"], g["V"], den=den, ckpt=ck), den, ck


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [s for s in SMALL if s[2] > 1])
@pytest.mark.parametrize("saved", ["out", "none", "out+den", "out+den+ckpt"])
def test_causal_backward_small(dt, shape, saved):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, dt, seed=21 + N, with_grad=True)
    g = _dev(x)
    O, den, ck = _saved(la, g, saved)
    dQ, dK, dV = la.la_backward_causal(g["Q"], g["K"], g["V"], g["G"], Out=O, Den=den, Ckpt=ck)
    torch.cuda.synchronize()
    RdQ, RdK, RdV = oracle.causal_backward_cumsum(x["Q"], x["K"], x["V"], x["G"])
    assert rel_err(dQ, RdQ) <= TOL[dt]
    assert rel_err(dK, RdK) <= TOL[dt]
    assert rel_err(dV, RdV) <= TOL[dt]


@pytest.mark.parametrize("shape", [
    (1, 2, 4096, 64, 64),     # few heads: one chunk per range
    (8, 40, 300, 64, 64),     # many short heads: ranges of several heads each, ragged tails
    (2, 3, 129, 64, 64),      # one chunk plus a single-token tail
    (1, 1, 128, 64, 64),
    (2, 3, 8300, 64, 64),     # several chunks per range, ranges crossing heads, ragged last chunk
])
@pytest.mark.parametrize("saved", ["out", "none", "out+den", "out+den+ckpt"])
def test_causal_backward_bf16_span_shapes(shape, saved):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "bf16", seed=23 + N, with_grad=True)
    g = _dev(x)
    O, den, ck = _saved(la, g, saved)
    dQ, dK, dV = la.la_backward_causal(g["Q"], g["K"], g["V"], g["G"], Out=O, Den=den, Ckpt=ck)
    la.la_check_device_status()
    idx = list(range(min(B * H, 6)))
    hs = [x[n].reshape(B * H, N, -1)[idx] for n in ("Q", "K", "V", "G")]
    RdQ, RdK, RdV = oracle.causal_backward_cumsum(*hs)
    assert rel_err(dQ.reshape(B * H, N, D)[idx], RdQ) <= TOL["bf16"]
    assert rel_err(dK.reshape(B * H, N, D)[idx], RdK) <= TOL["bf16"]
    assert rel_err(dV.reshape(B * H, N, M)[idx], RdV) <= TOL["bf16"]


@pytest.mark.parametrize("dt,M", [("f32", 32), ("bf16", 32), ("bf16", 64)])
@pytest.mark.parametrize("pass_out", [True, False])
def test_causal_backward_single_token(dt, M, pass_out):
    # N = 1: O_1 = V_1 whatever Q and K are, so dQ = dK = 0 exactly and dV = G.
    # The max-normalised error is undefined for an all-zero reference, so dQ
    # and dK are bounded against the natural scale max|G| * max|V| instead.
    la = _la()
    B, H, N, D = 2, 3, 1, 64
    x = synth.qkv(B, H, N, D, M, dt, seed=3, with_grad=True)
    g = _dev(x)
    O = la.la_forward_causal(g["Q"], g["K"], g["V"]) if pass_out else None
    dQ, dK, dV = la.la_backward_causal(g["Q"], g["K"], g["V"], g["G"], Out=O)
    torch.cuda.synchronize()
    scale = float(g["G"].float().abs().max() * g["V"].float().abs().max())
    assert float(dQ.float().abs().max()) <= TOL[dt] * 1e-2 * scale
    assert float(dK.float().abs().max()) <= TOL[dt] * 1e-2 * scale
    assert rel_err(dV, x["G"].double().numpy()) <= TOL[dt]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL)
def test_noncausal_small(dt, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, dt, seed=31 + N)
    g = _dev(x)
    O = la.la_forward_noncausal(g["Q"], g["K"], g["V"])
    torch.cuda.synchronize()
    Ro = oracle.noncausal_forward_assoc(x["Q"], x["K"], x["V"])[0]
    assert rel_err(O, Ro) <= TOL[dt]


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 64, 64),        # a single token
    (2, 3, 129, 64, 64),      # one chunk and a one-token tail
    (8, 40, 300, 64, 64),     # more heads than resident CTAs
    (1, 2, 4097, 64, 64),     # many spans per head, ragged tail
    (1, 1, 64, 64, 64),       # one 64-token stage
    (1, 1, 65, 64, 64),       # a one-token second stage
    (1, 2, 192, 64, 64),      # fewer stages than ring slots
    (2, 1, 448, 64, 64),      # more stages than ring slots: slots refilled
])
def test_noncausal_f32_tensor_core_shapes(shape):
    # fp32 at D = M = 64 runs on the tensor cores with operands split into two bf16 terms
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "f32", seed=37 + N)
    g = _dev(x)
    O = la.la_forward_noncausal(g["Q"], g["K"], g["V"])
    la.la_check_device_status()
    idx = list(range(min(B * H, 6)))
    hs = [x[n].reshape(B * H, N, -1)[idx] for n in ("Q", "K", "V")]
    Ro = oracle.noncausal_forward_assoc(*hs)[0]
    assert rel_err(O.reshape(B * H, N, M)[idx], Ro) <= TOL["f32"]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,D,M", [(2, 3, 64, 64), (1, 4, 32, 128), (3, 2, 128, 32)])
def test_decode_continues_prefill(dt, B, H, D, M):
    la = _la()
    N0, T = 150, 12
    x = synth.qkv(B, H, N0, D, M, dt, seed=41)
    g = _dev(x)
    _, S, Z = la.la_forward_causal(g["Q"], g["K"], g["V"], return_state=True)
    _, Rs, Rz = oracle.causal_forward_recurrent(x["Q"], x["K"], x["V"])
    for t in range(T):
        s = synth.decode_step_qkv(B, H, D, M, dt, seed=42, step=t)
        out = la.la_decode_step(s["q"].cuda(), s["k"].cuda(), s["v"].cuda(), S, Z)
        ro, Rs, Rz = oracle.decode_step(s["q"], s["k"], s["v"], Rs, Rz)
        torch.cuda.synchronize()
        assert rel_err(out, ro) <= TOL[dt]
    assert rel_err(S, Rs) <= TOL[dt] and rel_err(Z, Rz) <= TOL[dt]


def test_decode_rejects_bad_state_alignment():
    la = _la()
    q = torch.randn(1, 1, 64, device="cuda").bfloat16()
    S = torch.zeros(1 * 64 * 64 + 1, device="cuda")[1:].view(1, 1, 64, 64)
    Z = torch.zeros(1, 1, 64, device="cuda")
    with pytest.raises(la.LinAttnError, match="INVALID_ARG"):
        la.la_decode_step(q, q, q, S, Z)


# ------------------------------------------------------------ full sizes

def _sample_heads(BH, k=3):
    return sorted(set([0, BH // 2, BH - 1][:k]))


def _heads(t, idx):
    """[B,H,...] -> [len(idx), ...] for flat head indices."""
    return t.reshape((-1,) + tuple(t.shape[2:]))[idx]


def test_full_noncausal_f32():
    la = _la()
    w = synth.WORKLOADS["noncausal_f32"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale)
    g = _dev(x)
    O = la.la_forward_noncausal(g["Q"], g["K"], g["V"])
    torch.cuda.synchronize()
    idx = _sample_heads(w.B * w.H)
    Ro = oracle.noncausal_forward_assoc(_heads(x["Q"], idx), _heads(x["K"], idx), _heads(x["V"], idx))[0]
    assert rel_err(_heads(O, idx), Ro) <= TOL[w.dtype]
    # every row is a convex combination of all V rows of its head
    vmin = g["V"].amin(dim=2, keepdim=True)
    vmax = g["V"].amax(dim=2, keepdim=True)
    assert bool(((O >= vmin - 1e-4) & (O <= vmax + 1e-4)).all())


def test_full_causal_train_bf16():
    la = _la()
    w = synth.WORKLOADS["causal_train_bf16"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, with_grad=True)
    g = _dev(x)
    # the training step as the bench runs it: the forward keeps Out, the
    # normaliser and the state checkpoints, the backward takes them
    den = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    ck = torch.empty(la.la_causal_ckpt_floats(w.B, w.H, w.N, w.D, w.M), dtype=torch.float32,
                     device="cuda")
    O = la.la_forward_causal(g["Q"], g["K"], g["V"], den=den, ckpt=ck)
    dQ, dK, dV = la.la_backward_causal(g["Q"], g["K"], g["V"], g["G"], Out=O, Den=den, Ckpt=ck)
    torch.cuda.synchronize()
    idx = _sample_heads(w.B * w.H)
    hs = [_heads(x[n], idx) for n in ("Q", "K", "V", "G")]
    Ro, _, _, Rd = oracle.causal_forward_recurrent(*hs[:3], return_den=True)
    RdQ, RdK, RdV = oracle.causal_backward_cumsum(*hs)
    assert rel_err(_heads(O, idx), Ro) <= TOL[w.dtype]
    assert rel_err(_heads(den, idx), Rd) <= TOL[w.dtype]
    assert rel_err(_heads(dQ, idx), RdQ) <= TOL[w.dtype]
    assert rel_err(_heads(dK, idx), RdK) <= TOL[w.dtype]
    assert rel_err(_heads(dV, idx), RdV) <= TOL[w.dtype]
    # sum_j dV_j = sum_i G_i for every head (translation equivariance of O in V)
    lhs = dV.float().sum(dim=2)
    rhs = g["G"].float().sum(dim=2)
    assert float((lhs - rhs).abs().max() / rhs.abs().max()) <= 2e-2


def test_full_causal_long_bf16():
    la = _la()
    w = synth.WORKLOADS["causal_long_bf16"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale)
    g = _dev(x)
    O, S, Z = la.la_forward_causal(g["Q"], g["K"], g["V"], return_state=True)
    torch.cuda.synchronize()
    idx = [0, w.B * w.H - 1]
    Ro, Rs, Rz = oracle.causal_forward_recurrent(*[_heads(x[n], idx) for n in ("Q", "K", "V")])
    assert rel_err(_heads(O, idx), Ro) <= TOL[w.dtype]
    assert rel_err(_heads(S, idx), Rs) <= TOL[w.dtype]
    assert rel_err(_heads(Z, idx), Rz) <= TOL[w.dtype]
    # prefix convex hull at any size: min_{j<=i} V_j <= O_i <= max_{j<=i} V_j
    V = g["V"].float()
    lo = torch.cummin(V, dim=2).values
    hi = torch.cummax(V, dim=2).values
    slack = 2e-2 * float(V.abs().max())
    assert bool(((O.float() >= lo - slack) & (O.float() <= hi + slack)).all())


def test_full_decode_bf16():
    la = _la()
    w = synth.WORKLOADS["decode_bf16"]
    B, H, D, M = w.B, w.H, w.D, w.M
    x = synth.qkv(B, H, w.prefill, D, M, w.dtype, w.seed, w.scale)
    g = _dev(x)
    _, S, Z = la.la_forward_causal(g["Q"], g["K"], g["V"], return_state=True)
    idx = _sample_heads(B * H)
    _, Rs, Rz = oracle.causal_forward_recurrent(*[_heads(x[n], idx) for n in ("Q", "K", "V")])
    torch.cuda.synchronize()
    assert rel_err(_heads(S, idx), Rs) <= TOL[w.dtype]
    # every step's output on the sampled heads, gathered on the device and compared at the end
    got = torch.empty((w.steps, len(idx), M), dtype=torch.float32, device="cuda")
    ref = np.empty((w.steps, len(idx), M))
    idx_dev = torch.tensor(idx, device="cuda")
    for t in range(w.steps):
        s = synth.decode_step_qkv(B, H, D, M, w.dtype, w.seed, t)
        out = la.la_decode_step(s["q"].cuda(non_blocking=True), s["k"].cuda(non_blocking=True),
                                s["v"].cuda(non_blocking=True), S, Z)
        got[t] = out.reshape(B * H, M).index_select(0, idx_dev)
        hq = [s[n].reshape(B * H, -1)[idx] for n in ("q", "k", "v")]
        ref[t], Rs, Rz = oracle.decode_step(*hq, Rs, Rz)
    torch.cuda.synchronize()
    worst = max(rel_err(got[t], ref[t]) for t in range(w.steps))
    assert worst <= TOL[w.dtype]
    assert rel_err(_heads(S, idx), Rs) <= TOL[w.dtype]
    assert rel_err(_heads(Z, idx), Rz) <= TOL[w.dtype]
