"""GPU parity of la_backward_noncausal (through the C ABI) against the fp64 oracle.

The gradient of the non-causal form ("Transformers are RNNs" section 二,
eq. linear) by the cumulative-sum formulas of section 三（一）4 with full sums,
and the quotient rule for the denominator.  Error measure and tolerances as in
test_gpu_parity: max|got - ref| / max|ref| per tensor, 1e-4 (fp32), 2e-2 (bf16).
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
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


SHAPES = [(1, 1, 256, 32, 32), (2, 3, 200, 64, 32), (1, 2, 517, 128, 64), (2, 2, 1000, 64, 64),
          (1, 2, 130, 32, 128), (1, 3, 77, 128, 128), (3, 1, 2049, 64, 128), (2, 2, 4097, 64, 64)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("pass_out", [True, False])
def test_noncausal_backward_small(dt, shape, pass_out):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, dt, seed=90 + N, with_grad=True)
    g = {k: v.cuda() for k, v in x.items()}
    O = la.la_forward_noncausal(g["Q"], g["K"], g["V"]) if pass_out else None
    dQ, dK, dV = la.la_backward_noncausal(g["Q"], g["K"], g["V"], g["G"], Out=O)
    la.la_check_device_status()
    R = oracle.noncausal_backward_assoc(x["Q"], x["K"], x["V"], x["G"])
    for name, got, ref in zip(("dQ", "dK", "dV"), (dQ, dK, dV), R):
        assert rel_err(got, ref) <= TOL[dt], name


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_noncausal_backward_single_token_and_empty(dt):
    la = _la()
    x = synth.qkv(2, 3, 1, 64, 64, dt, seed=95, with_grad=True)
    g = {k: v.cuda() for k, v in x.items()}
    dQ, dK, dV = la.la_backward_noncausal(g["Q"], g["K"], g["V"], g["G"])
    la.la_check_device_status()
    # one token: O_1 = V_1, so dQ = dK = 0 and dV = G
    scale = float(g["G"].float().abs().max() * g["V"].float().abs().max())
    assert float(dQ.float().abs().max()) <= TOL[dt] * 1e-2 * scale
    assert float(dK.float().abs().max()) <= TOL[dt] * 1e-2 * scale
    assert rel_err(dV, x["G"].double().numpy()) <= TOL[dt]
    e = torch.empty((2, 3, 0, 64), dtype=g["Q"].dtype, device="cuda")
    la.la_backward_noncausal(e, e, e, e)  # no work, no error


def test_full_noncausal_backward_f32():
    # the non-causal workload's shape: B=8 H=8 N=4096 D=M=64, fp32
    la = _la()
    w = synth.WORKLOADS["noncausal_f32"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, with_grad=True)
    g = {k: v.cuda() for k, v in x.items()}
    O = la.la_forward_noncausal(g["Q"], g["K"], g["V"])
    dQ, dK, dV = la.la_backward_noncausal(g["Q"], g["K"], g["V"], g["G"], Out=O)
    la.la_check_device_status()
    BH = w.B * w.H
    idx = [0, BH // 2, BH - 1]
    hs = [x[n].reshape(BH, w.N, -1)[idx] for n in ("Q", "K", "V", "G")]
    R = oracle.noncausal_backward_assoc(*hs)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dQ, dK, dV), R):
        assert rel_err(got.reshape(BH, w.N, -1)[idx], ref) <= TOL[w.dtype], name
    # at any size: sum_j dV_j = sum_i G_i per head (O moves with a shift of every V row)
    lhs, rhs = dV.double().sum(dim=2), g["G"].double().sum(dim=2)
    assert float((lhs - rhs).abs().max() / rhs.abs().max()) <= 1e-4
