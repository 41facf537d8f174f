"""la_forward_noncausal_noalloc: the non-causal forward for callers that may
not allocate device memory inside an op (their device memory is planned ahead
by a host framework, or allocation is forbidden or too slow where they run).
Its scratch is a fixed device array inside the library, shared by all calls.

Checked through the C ABI (ctypes) against la_forward_noncausal and against
the fp64 oracle, twice in a row with different inputs, so that scratch left
behind by the first call cannot leak into the second; and the device's free
memory is checked unchanged across a call.  This file is collected last on
purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from linear_attention_02_gb300 import _native, synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DT = {"f32": _native.LA_DTYPE_F32, "bf16": _native.LA_DTYPE_BF16}


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _call(fn, x, out, shape, dt):
    B, H, N, D, M = shape
    st = torch.cuda.current_stream().cuda_stream
    return fn(x["Q"].data_ptr(), x["K"].data_ptr(), x["V"].data_ptr(), out.data_ptr(), B, H, N, D, M,
              DT[dt], ctypes.c_void_p(st))


# (1, 127, 300, 128, 128): 127 heads leave room for one span per head in the
# fixed scratch, so the call takes the branch that lengthens the spans.
@pytest.mark.parametrize("dt,shape", [("f32", (8, 8, 4096, 64, 64)),
                                      ("bf16", (2, 3, 517, 128, 64)),
                                      ("f32", (1, 2, 77, 32, 128)),
                                      ("bf16", (1, 127, 300, 128, 128))])
def test_noalloc_matches_allocating_entry_point(dt, shape):
    lib = _native.lib
    B, H, N, D, M = shape
    for call in range(2):
        xc = synth.qkv(B, H, N, D, M, dt, seed=500 + call)
        x = {k: v.cuda() for k, v in xc.items()}
        ref = torch.empty((B, H, N, M), dtype=x["V"].dtype, device="cuda")
        got = torch.full_like(ref, float("nan"))
        assert _call(lib.la_forward_noncausal, x, ref, shape, dt) == _native.LA_OK
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        assert _call(lib.la_forward_noncausal_noalloc, x, got, shape, dt) == _native.LA_OK, \
            lib.la_last_error_message()
        torch.cuda.synchronize()
        if call == 1:  # the first call may commit the fixed array; later ones take nothing
            assert torch.cuda.mem_get_info()[0] == free0
        assert _rel(got, ref) <= TOL[dt], f"call {call}"
        # against the oracle on a few heads (all of them when small)
        hs = list(range(min(B * H, 4)))
        Q = xc["Q"].reshape(B * H, N, D)[hs]
        K = xc["K"].reshape(B * H, N, D)[hs]
        V = xc["V"].reshape(B * H, N, M)[hs]
        want = oracle.noncausal_forward_assoc(Q, K, V)[0]
        assert _rel(got.reshape(B * H, N, M)[hs], torch.from_numpy(want)) <= TOL[dt], f"call {call}"


def test_noalloc_rejects_work_beyond_its_scratch():
    lib = _native.lib
    # B*H = 128 heads at D = M = 128 need 2 * 128 * 16512 * 4 bytes > 16 MiB
    x = {k: v.cuda() for k, v in synth.qkv(1, 128, 8, 128, 128, "bf16", seed=1).items()}
    out = torch.empty((1, 128, 8, 128), dtype=torch.bfloat16, device="cuda")
    assert _call(lib.la_forward_noncausal_noalloc, x, out, (1, 128, 8, 128, 128), "bf16") == \
        _native.LA_ERR_INVALID_ARG
    assert b"fixed scratch" in lib.la_last_error_message()
