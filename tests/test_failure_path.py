"""The device error word: bounded waits that expire are reported, and the device stays usable.

A self-test kernel waits on an mbarrier phase that nothing completes and on a
flag that nothing sets, each for a few thousand polls; both give up and set
their bits in the error word, exactly as the library's kernels do when a copy,
a product or a look-back flag never arrives.  Nothing faults or hangs.
"""
import pytest
import torch

import oracle
from linear_attention_02_gb300 import _native, synth

pytestmark = pytest.mark.gpu


def test_expired_waits_are_reported_and_the_device_stays_usable():
    import linear_attention_02_gb300 as la
    la.la_check_device_status()  # nothing pending before
    la.la_selftest_expired_waits()
    with pytest.raises(la.LinAttnError) as e:
        la.la_check_device_status()
    assert e.value.status == _native.LA_ERR_TIMEOUT
    assert "0x3" in str(e.value)  # both the mbarrier wait and the flag wait gave up
    la.la_check_device_status()  # the check cleared the word

    B, H, N, D, M = 1, 2, 300, 64, 64  # the device still computes correctly
    x = synth.qkv(B, H, N, D, M, "bf16", seed=5)
    O = la.la_forward_causal(*(x[n].cuda() for n in ("Q", "K", "V")))
    la.la_check_device_status()
    Ro, _, _ = oracle.causal_forward_recurrent(x["Q"], x["K"], x["V"])
    err = float((O.float().cpu().double() - torch.as_tensor(Ro)).abs().max() / abs(Ro).max())
    assert err <= 2e-2


def _timed_out(la):
    with pytest.raises(la.LinAttnError) as e:
        la.la_check_device_status()
    assert e.value.status == _native.LA_ERR_TIMEOUT
    return str(e.value)


def test_withheld_lookback_flag_times_out_in_the_forward_kernel():
    # 1 head of 64 chunks: every chunk is a unit of the tensor-core forward's split, units
    # 1 .. 63 look back to unit 0, which (test hook) does not publish; their waits give up
    # after 2000 polls, set the look-back bit (0x2), drain their copies and end
    import linear_attention_02_gb300 as la
    la.la_check_device_status()
    x = synth.qkv(1, 1, 64 * 128, 64, 64, "bf16", seed=9)
    g = {k: v.cuda() for k, v in x.items()}
    assert _native.lib.la_debug_withhold_publication(0, 2000) == _native.LA_OK
    la.la_forward_causal(g["Q"], g["K"], g["V"])
    assert "0x2" in _timed_out(la)
    la.la_check_device_status()  # cleared
    # the same call without the hook is correct on the same device
    O = la.la_forward_causal(g["Q"], g["K"], g["V"])
    la.la_check_device_status()
    Ro, _, _ = oracle.causal_forward_recurrent(x["Q"], x["K"], x["V"])
    err = float((O.float().cpu().double() - torch.as_tensor(Ro)).abs().max() / abs(Ro).max())
    assert err <= 2e-2


def test_withheld_lookback_flag_times_out_in_the_backward_kernel():
    # without checkpoints the backward's prefix kernel finds each range's starting state by
    # the same look-back; unit 0 of its split (one head, 64 chunks over 152 units) withholds
    import linear_attention_02_gb300 as la
    la.la_check_device_status()
    x = synth.qkv(1, 1, 64 * 128, 64, 64, "bf16", seed=10, with_grad=True)
    g = {k: v.cuda() for k, v in x.items()}
    O = la.la_forward_causal(g["Q"], g["K"], g["V"])
    la.la_check_device_status()
    assert _native.lib.la_debug_withhold_publication(0, 2000) == _native.LA_OK
    la.la_backward_causal(g["Q"], g["K"], g["V"], g["G"], Out=O)
    assert "0x2" in _timed_out(la)
    dQ, dK, dV = la.la_backward_causal(g["Q"], g["K"], g["V"], g["G"], Out=O)
    la.la_check_device_status()
    R = oracle.causal_backward_cumsum(x["Q"], x["K"], x["V"], x["G"])
    for got, ref in zip((dQ, dK, dV), R):
        err = float((got.float().cpu().double() - torch.as_tensor(ref)).abs().max() / abs(ref).max())
        assert err <= 2e-2


def test_hook_rejects_bad_arguments():
    assert _native.lib.la_debug_withhold_publication(-1, 10) == _native.LA_ERR_INVALID_ARG
    assert _native.lib.la_debug_withhold_publication(0, 0) == _native.LA_ERR_INVALID_ARG
