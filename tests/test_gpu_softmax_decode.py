"""GPU parity of la_softmax_decode_step (the KV-cache comparator of the
recurrent decode step) against the fp64 oracle, through the C ABI.

Standard Transformer inference ("Transformer与RNN的深层联结", section 2): the
step's k, v are appended to the cache, then out = softmax(q K^T / sqrt(D)) V.
Checked: the output, that the new row landed in the cache, successive steps
growing the cache, an empty cache, and the decode workload's shape at a full
cache (256 sequences x 16 heads, 4096 positions) on sampled heads.
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


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,D,T,T_max", [(2, 3, 64, 0, 8), (1, 2, 32, 1, 2), (2, 2, 128, 300, 301),
                                           (1, 4, 64, 1000, 1500), (3, 1, 32, 777, 800)])
def test_softmax_decode_small(dt, B, H, D, T, T_max):
    la = _la()
    c = synth.qkv(B, H, T_max, D, D, dt, seed=100 + T)       # cache contents (rows >= T unused)
    s = synth.decode_step_qkv(B, H, D, D, dt, seed=101, step=T)
    Kc, Vc = c["K"].cuda(), c["V"].cuda()
    out = la.la_softmax_decode_step(s["q"].cuda(), s["k"].cuda(), s["v"].cuda(), Kc, Vc, T)
    la.la_check_device_status()
    ref = oracle.softmax_decode_step(s["q"], s["k"], s["v"], c["K"][:, :, :T], c["V"][:, :, :T])
    assert rel_err(out, ref) <= TOL[dt]
    # the step's own row is now in the cache; nothing else changed
    assert torch.equal(Kc[:, :, T].cpu(), s["k"]) and torch.equal(Vc[:, :, T].cpu(), s["v"])
    assert torch.equal(Kc[:, :, :T].cpu(), c["K"][:, :, :T])


def test_softmax_decode_successive_steps():
    la = _la()
    B, H, D, T0, steps, dt = 2, 3, 64, 50, 20, "bf16"
    c = synth.qkv(B, H, T0 + steps, D, D, dt, seed=102)
    Kc, Vc = c["K"].cuda(), c["V"].cuda()
    Kref, Vref = c["K"][:, :, :T0].clone(), c["V"][:, :, :T0].clone()
    for t in range(steps):
        s = synth.decode_step_qkv(B, H, D, D, dt, seed=103, step=t)
        out = la.la_softmax_decode_step(s["q"].cuda(), s["k"].cuda(), s["v"].cuda(), Kc, Vc, T0 + t)
        ref = oracle.softmax_decode_step(s["q"], s["k"], s["v"], Kref, Vref)
        torch.cuda.synchronize()
        assert rel_err(out, ref) <= TOL[dt], t
        Kref = torch.cat([Kref, s["k"][:, :, None]], 2)
        Vref = torch.cat([Vref, s["v"][:, :, None]], 2)


def test_softmax_decode_full_cache():
    # the decode workload's heads (256 sequences x 16, D = M = 64) with a full
    # 4096-position cache (2048 prefill + 2048 steps); sampled heads vs the oracle
    la = _la()
    w = synth.WORKLOADS["decode_bf16"]
    B, H, D, T_max = w.B, w.H, w.D, w.prefill + w.steps
    T = T_max - 1
    Kc = synth.randn((B, H, T_max, D), "bf16", 104, device="cuda")
    Vc = synth.randn((B, H, T_max, D), "bf16", 105, device="cuda")
    s = synth.decode_step_qkv(B, H, D, D, "bf16", seed=106, step=0)
    out = la.la_softmax_decode_step(s["q"].cuda(), s["k"].cuda(), s["v"].cuda(), Kc, Vc, T)
    la.la_check_device_status()
    BH = B * H
    idx = [0, BH // 2, BH - 1]
    Kh = Kc.reshape(BH, T_max, D)[idx, :T].cpu()
    Vh = Vc.reshape(BH, T_max, D)[idx, :T].cpu()
    hq = [s[n].reshape(BH, D)[idx] for n in ("q", "k", "v")]
    ref = oracle.softmax_decode_step(*hq, Kh, Vh)
    assert rel_err(out.reshape(BH, D)[idx], ref) <= TOL["bf16"]
    # every output is a convex combination of its head's value rows
    V = Vc.float()
    assert bool((out >= V.amin(dim=2) - 1e-3).all() and (out <= V.amax(dim=2) + 1e-3).all())


def test_softmax_decode_rejects_bad_arguments():
    la = _la()
    q = torch.zeros(1, 1, 64, device="cuda", dtype=torch.bfloat16)
    Kc = torch.zeros(1, 1, 4, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(la.LinAttnError, match="INVALID_ARG"):
        la.la_softmax_decode_step(q, q, q, Kc, Kc, 4)
    v32 = torch.zeros(1, 1, 32, device="cuda", dtype=torch.bfloat16)
    V32 = torch.zeros(1, 1, 4, 32, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(la.LinAttnError, match="UNSUPPORTED"):
        la.la_softmax_decode_step(q, q, v32, Kc, V32, 1)
