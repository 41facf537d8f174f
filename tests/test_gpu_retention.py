"""GPU parity of the retention entry points (linear attention with decay,
"Transformer and Variants" sections 1.3.2 and 1.3.4) against the fp64 oracle,
through the C ABI: decay 1 (the unnormalised form), RetNet (one decay per
head) and gated retention (one decay per token), the forward with carried
state and the decode step.  Errors are max|got - ref| / max|ref| per tensor:
1e-4 for fp32 storage, 2e-2 for bf16 storage.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
KINDS = ["decay1", "retnet", "gated"]


def _la():
    import linear_attention_02_gb300 as la
    return la


def rel_err(got, ref) -> float:
    got = np.asarray(got.float().cpu().numpy() if isinstance(got, torch.Tensor) else got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def _decay_kw(kind, B, H, N, seed):
    if kind == "retnet":
        return {"gamma_head": synth.decays((H,), seed, 0.9, 1.0)}
    if kind == "gated":
        return {"gates": synth.decays((B, H, N), seed, 0.85, 1.0)}
    return {}


SHAPES = [(1, 1, 256, 32, 32), (2, 3, 200, 64, 32), (1, 2, 517, 128, 64), (2, 2, 1000, 64, 64),
          (1, 2, 130, 32, 128), (1, 1, 1, 64, 64), (1, 3, 77, 128, 128), (2, 2, 2049, 64, 64)]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_retention_forward_small(kind, dt, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, dt, seed=120 + N)
    kw = _decay_kw(kind, B, H, N, seed=121)
    O, S = la.la_forward_retention(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(),
                                   **{k: v.cuda() for k, v in kw.items()}, return_state=True)
    la.la_check_device_status()
    Ro, Rs = oracle.retention_forward_recurrent(x["Q"], x["K"], x["V"], **kw)
    assert rel_err(O, Ro) <= TOL[dt]
    assert rel_err(S, Rs) <= TOL[dt]


@pytest.mark.parametrize("kind", KINDS)
def test_retention_carried_state_and_decode(kind):
    la = _la()
    B, H, N, D, M, cut, dt = 2, 3, 700, 64, 64, 333, "bf16"
    x = synth.qkv(B, H, N, D, M, dt, seed=122)
    kw = _decay_kw(kind, B, H, N, seed=123)
    g = {k: v.cuda() for k, v in x.items()}
    kwd = {k: v.cuda() for k, v in kw.items()}
    part = lambda a, b: {k: (v[:, :, a:b].contiguous() if k == "gates" else v) for k, v in kwd.items()}
    Oa, Sa = la.la_forward_retention(*(g[n][:, :, :cut].contiguous() for n in "QKV"), **part(0, cut),
                                     return_state=True)
    Ob, Sb = la.la_forward_retention(*(g[n][:, :, cut:].contiguous() for n in "QKV"), **part(cut, N),
                                     S_init=Sa, return_state=True)
    la.la_check_device_status()
    Ro, Rs = oracle.retention_forward_recurrent(x["Q"], x["K"], x["V"], **kw)
    assert rel_err(torch.cat([Oa, Ob], 2), Ro) <= TOL[dt]
    assert rel_err(Sb, Rs) <= TOL[dt]
    # decode steps continue the forward's state
    S = Sb.clone()
    RS = Rs
    for t in range(6):
        s = synth.decode_step_qkv(B, H, D, M, dt, seed=124, step=t)
        if kind == "gated":
            gate = synth.decays((B, H), 125 + t, 0.85, 1.0)
            dkw, ogam = {"gate": gate.cuda()}, gate
        elif kind == "retnet":
            dkw, ogam = {"gamma_head": kwd["gamma_head"]}, kw["gamma_head"][None, :].expand(B, H)
        else:
            dkw, ogam = {}, torch.ones(B, H)
        out = la.la_retention_decode_step(s["q"].cuda(), s["k"].cuda(), s["v"].cuda(), S, **dkw)
        ro, RS = oracle.retention_decode_step(s["q"], s["k"], s["v"], ogam.double().numpy(), RS)
        torch.cuda.synchronize()
        assert rel_err(out, ro) <= TOL[dt], t
    assert rel_err(S, RS) <= TOL[dt]


def test_retention_full_gated_bf16():
    # the training workload's shape, gated: B=4 H=16 N=8192 D=M=64, bf16
    la = _la()
    w = synth.WORKLOADS["causal_train_bf16"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale)
    gates = synth.decays((w.B, w.H, w.N), w.seed + 5, 0.85, 1.0)
    O, S = la.la_forward_retention(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(), gates=gates.cuda(),
                                   return_state=True)
    la.la_check_device_status()
    BH = w.B * w.H
    idx = [0, BH // 2, BH - 1]
    hs = [x[n].reshape(BH, w.N, -1)[idx][None] for n in ("Q", "K", "V")]
    Ro, Rs = oracle.retention_forward_recurrent(*hs, gates=gates.reshape(BH, w.N)[idx][None])
    assert rel_err(O.reshape(BH, w.N, -1)[idx], Ro[0]) <= TOL[w.dtype]
    assert rel_err(S.reshape(BH, w.D, w.M)[idx], Rs[0]) <= TOL[w.dtype]


def test_retention_rejects_both_decays():
    la = _la()
    x = torch.zeros(1, 2, 8, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        la.la_forward_retention(x, x, x, gamma_head=torch.ones(2, device="cuda"),
                                gates=torch.ones(1, 2, 8, device="cuda"))


# bf16 with D = M in {64, 128} runs the tensor-core kernel: the chunks of all heads cut
# into equal ranges, so a range can hold the tail of one head and the start of
# another, or stop inside a head (its aggregate then carries the piece's total decay)
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(8, 40, 300, 64, 64), (1, 2, 5000, 128, 128), (2, 3, 8300, 64, 64),
                                   (1, 1, 128, 64, 64), (2, 3, 129, 64, 64), (1, 1, 20000, 64, 64)])
def test_retention_tensor_core_ranges(kind, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "bf16", seed=126 + N)
    kw = _decay_kw(kind, B, H, N, seed=127)
    S0 = torch.randn(B, H, D, M) * 0.1
    O, S = la.la_forward_retention(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(),
                                   **{k: v.cuda() for k, v in kw.items()}, S_init=S0.cuda(),
                                   return_state=True)
    la.la_check_device_status()
    idx = list(range(min(B * H, 6)))
    hs = [x[n].reshape(B * H, N, -1)[idx][None] for n in ("Q", "K", "V")]
    okw = {}
    if kind == "retnet":
        okw["gamma_head"] = kw["gamma_head"].repeat(B)[idx]
    elif kind == "gated":
        okw["gates"] = kw["gates"].reshape(B * H, N)[idx][None]
    Ro, Rs = oracle.retention_forward_recurrent(*hs, S0=S0.reshape(B * H, D, M)[idx][None], **okw)
    assert rel_err(O.reshape(B * H, N, M)[idx], Ro[0]) <= TOL["bf16"]
    assert rel_err(S.reshape(B * H, D, M)[idx], Rs[0]) <= TOL["bf16"]


# Chunks whose total log2 decay is at least -100 fold their decays into the Q and K rows
# (P comes out decayed); stronger ones take P's decay element by element.  Gates in
# [0.25, 1) put about half the chunks on each side of that line; gates near 1e-25
# are clamped to 2^-64 per token, far past it.
@pytest.mark.parametrize("gate_range", [(0.25, 1.0), (1e-30, 1e-20)])
@pytest.mark.parametrize("shape", [(2, 3, 2049, 64, 64), (1, 2, 1000, 128, 128)])
def test_retention_tensor_core_strong_decays(gate_range, shape):
    la = _la()
    B, H, N, D, M = shape
    x = synth.qkv(B, H, N, D, M, "bf16", seed=160 + N)
    gates = synth.decays((B, H, N), 161, *gate_range)
    S0 = torch.randn(B, H, D, M) * 0.1
    O, S = la.la_forward_retention(x["Q"].cuda(), x["K"].cuda(), x["V"].cuda(), gates=gates.cuda(),
                                   S_init=S0.cuda(), return_state=True)
    la.la_check_device_status()
    idx = list(range(min(B * H, 4)))
    hs = [x[n].reshape(B * H, N, -1)[idx][None] for n in ("Q", "K", "V")]
    Ro, Rs = oracle.retention_forward_recurrent(*hs, S0=S0.reshape(B * H, D, M)[idx][None],
                                                gates=gates.reshape(B * H, N)[idx][None])
    assert rel_err(O.reshape(B * H, N, M)[idx], Ro[0]) <= TOL["bf16"]
    assert rel_err(S.reshape(B * H, D, M)[idx], Rs[0]) <= TOL["bf16"]
