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
