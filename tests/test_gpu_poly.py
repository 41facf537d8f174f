"""GPU parity of la_forward_poly2 (attention with the degree-2 polynomial
similarity (q . k)^2 through its explicit feature map, "Transformers are
RNNs" section 二 (3)) against the fp64 oracle, through the C ABI: causal and
over all tokens, both dtypes, ragged chunks and spans, one token, and a full
workload on sampled heads.  Errors: max|got - ref| / max|ref| per tensor,
1e-4 for fp32 storage, 2e-2 for bf16 storage."""
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


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 32, 32), (1, 2, 64, 32, 64), (2, 3, 200, 32, 32),
                                   (1, 2, 1000, 32, 64), (2, 1, 2049, 32, 32)])
def test_poly2_small(causal, dt, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, dt, seed=140 + N)
    O = la.la_forward_poly2(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(), causal=causal)
    la.la_check_device_status()
    ref = oracle.poly_forward_state(x["Q"], x["K"], x["V"], causal)
    assert rel_err(O, ref) <= TOL[dt]


# bf16 with M = 64 runs the tensor-core kernel: four CTAs per head, each owning two
# 128-feature slices of the D^2 = 1024 features, partial rows added into an fp32
# accumulator; one token, a chunk and one token, ragged multi-chunk heads
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 1, 1, 32, 64), (1, 1, 129, 32, 64), (2, 3, 300, 32, 64),
                                   (1, 2, 2049, 32, 64)])
def test_poly2_tensor_core(causal, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "bf16", seed=150 + N)
    O = la.la_forward_poly2(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(), causal=causal)
    la.la_check_device_status()
    ref = oracle.poly_forward_state(x["Q"], x["K"], x["V"], causal)
    assert rel_err(O, ref) <= TOL["bf16"]


# inputs off centre and scaled (q, k ~ N(-1, 2^2)): features x_a x_b of either sign and a
# wide range, normalisers far from 1
@pytest.mark.parametrize("causal", [True, False])
def test_poly2_tensor_core_wide_inputs(causal):
    la = _la()
    B, H, N, D, M = 1, 2, 700, 32, 64
    x = synth.qkv(B, H, N, D, M, "bf16", seed=157, scale=2.0, qk_mean=-1.0)
    O = la.la_forward_poly2(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(), causal=causal)
    la.la_check_device_status()
    ref = oracle.poly_forward_state(x["Q"], x["K"], x["V"], causal)
    assert rel_err(O, ref) <= TOL["bf16"]


def test_poly2_full_bf16():
    # B=4 H=16 N=4096 D=32 M=64, bf16: two heads against the oracle, every head's
    # rows inside the convex hull of the values it sees
    la = _la()
    B, H, N, D, M = 4, 16, 4096, 32, 64
    x = synth.qkv(B, H, N, D, M, "bf16", seed=141)
    g = {k: v.cuda() for k, v in x.items()}
    O = la.la_forward_poly2(g["Q"], g["K"], g["V"], causal=True)
    la.la_check_device_status()
    idx = [0, B * H - 1]
    hs = [x[n].reshape(B * H, N, -1)[idx] for n in ("Q", "K", "V")]
    assert rel_err(O.reshape(B * H, N, M)[idx], oracle.poly_forward_state(*hs, True)) <= TOL["bf16"]
    V = g["V"].float()
    lo, hi = torch.cummin(V, dim=2).values, torch.cummax(V, dim=2).values
    slack = 2e-2 * float(V.abs().max())
    assert bool(((O.float() >= lo - slack) & (O.float() <= hi + slack)).all())


def test_poly2_rejects_other_head_sizes():
    la = _la()
    x = torch.zeros(1, 1, 8, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(la.LinAttnError, match="UNSUPPORTED"):
        la.la_forward_poly2(x, x, x)
