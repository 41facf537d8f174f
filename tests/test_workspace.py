"""la_workspace_bytes: the scratch each call takes from the library's pool.

On the host the sizes are checked against hand-computed values for the
workloads (with the SM count given, the function is pure arithmetic); on the
GPU every op's actual peak pool use (la_scratch_peak_bytes) is checked against
the reported size."""
import ctypes

import pytest
import torch

from linear_attention_02_gb300 import _native

F32, BF16 = _native.LA_DTYPE_F32, _native.LA_DTYPE_BF16
SAVED_ALL = _native.LA_SAVED_OUT | _native.LA_SAVED_DEN | _native.LA_SAVED_CKPT


def _ws(op, B, H, N, D, M, dt, saved=0, sms=152):
    return _native.lib.la_workspace_bytes(op.encode(), B, H, N, D, M, dt, saved, sms)


def test_training_forward_bytes():
    # bf16 D = M = 64: two CTAs per SM -> 304 slots; 64 heads x 64 chunks = 4096
    # chunks cut into ranges of ceil(4096 / 304) = 14 -> 293 units; each unit
    # publishes two (S | Z) states of 64*64 + 64 floats (its piece's aggregate and the
    # head's state at the piece's end), plus one flag per unit and the ticket, plus
    # 256 bytes of slack.
    units = 293
    want = 2 * 4 * units * (64 * 64 + 64) + 4 * (units + 1) + 256
    assert _ws("la_forward_causal", 4, 16, 8192, 64, 64, BF16) == want


def test_training_backward_bytes():
    # one CTA per SM -> 152 slots; ranges of ceil(4096 / 152) = 27 chunks -> 152
    # units.  Two state arrays (S and R shares), flags, bf16 gn rows [64][8192][64],
    # fp32 gd rows [64][8192]; each part rounded up to 256 bytes.
    up = lambda x: (x + 255) // 256 * 256
    agg = 4 * 152 * (64 * 64 + 64)
    want = 2 * up(agg) + up(4 * 153) + up(2 * 64 * 8192 * 64) + up(4 * 64 * 8192)
    assert _ws("la_backward_causal", 4, 16, 8192, 64, 64, BF16, SAVED_ALL) == want
    # without Out the call recomputes the forward: its output tile, normaliser,
    # checkpoints (8 slots per head) and the forward's own scratch on top
    fwd = _ws("la_forward_causal", 4, 16, 8192, 64, 64, BF16)
    ck = 4 * 64 * 8 * (64 * 64 + 64)
    assert _ws("la_backward_causal", 4, 16, 8192, 64, 64, BF16, 0) == \
        want + up(2 * 64 * 8192 * 64) + up(4 * 64 * 8192) + up(ck) + fwd


def test_noncausal_and_decode_bytes():
    # fp32 D = M = 64, 64 heads x 32 chunks: 4 spans per head (ranges of 8 chunks,
    # 256 state CTAs in one wave of 304), one (S | Z) partial per span
    assert _ws("la_forward_noncausal", 8, 8, 4096, 64, 64, F32) == 4 * 64 * 4 * (64 * 64 + 64)
    assert _ws("la_decode_step", 256, 16, 0, 64, 64, BF16) == 0
    assert _ws("la_forward_noncausal_noalloc", 8, 8, 4096, 64, 64, F32) == 0


def test_cuda_core_paths_bytes():
    # fp32 causal D = M = 32: chunks of 64, spans = min(ceil(2*152 / 1), 4) = 4 for N = 256
    assert _ws("la_forward_causal", 1, 1, 256, 32, 32, F32) == 4 * 4 * (32 * 32 + 32)
    # one span (BH large): no aggregates at all
    assert _ws("la_forward_causal", 1, 400, 256, 32, 32, F32) == 0


def test_poly2_bytes():
    # bf16, M = 64: the tensor-core path's fp32 [numerator | normaliser | 15 copies]
    # accumulator, 80 floats per token and head
    assert _ws("la_forward_poly2", 4, 16, 4096, 32, 64, BF16) == 4 * 64 * 4096 * 80
    # other shapes on the CUDA cores: span aggregates of the 528 features and the accumulator
    assert _ws("la_forward_poly2", 1, 2, 1000, 32, 32, F32) > 0
    assert _ws("la_forward_poly2", 1, 2, 1000, 64, 64, BF16) == _native.SIZE_MAX


def test_bad_queries():
    lib = _native.lib
    assert _ws("la_forward_sideways", 1, 1, 8, 64, 64, F32) == _native.SIZE_MAX
    assert b"unknown op" in lib.la_last_error_message()
    assert _ws("la_forward_causal", 1, 1, 8, 48, 64, F32) == _native.SIZE_MAX
    assert _ws("la_forward_causal", -1, 1, 8, 64, 64, F32) == _native.SIZE_MAX
    assert _ws("la_forward_causal", 0, 1, 8, 64, 64, F32) == 0


def _peak_of(fn):
    import linear_attention_02_gb300 as la
    torch.cuda.synchronize()
    la.la_scratch_peak_bytes(reset=True)
    fn()
    torch.cuda.synchronize()
    return la.la_scratch_peak_bytes()


@pytest.mark.gpu
@pytest.mark.parametrize("dt,shape", [("bf16", (2, 3, 1100, 64, 64)), ("bf16", (1, 2, 700, 128, 128)),
                                      ("f32", (2, 2, 600, 64, 64)), ("f32", (1, 3, 333, 32, 128))])
def test_peak_pool_use_matches_report(dt, shape):
    import linear_attention_02_gb300 as la
    from linear_attention_02_gb300 import synth
    B, H, N, D, M = shape
    x = {k: v.cuda() for k, v in synth.qkv(B, H, N, D, M, dt, seed=31, with_grad=True).items()}
    tdt = x["Q"].dtype
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    den = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ck = torch.empty(la.la_causal_ckpt_floats(B, H, N, D, M), dtype=torch.float32, device="cuda")
    out = {}

    def fwd():
        out["O"] = la.la_forward_causal(x["Q"], x["K"], x["V"], den=den, ckpt=ck)

    cases = [("la_forward_causal", 0, fwd),
             ("la_backward_causal", SAVED_ALL,
              lambda: la.la_backward_causal(x["Q"], x["K"], x["V"], x["G"], Out=out["O"], Den=den,
                                            Ckpt=ck)),
             ("la_backward_causal", 0, lambda: la.la_backward_causal(x["Q"], x["K"], x["V"], x["G"])),
             ("la_forward_noncausal", 0, lambda: la.la_forward_noncausal(x["Q"], x["K"], x["V"]))]
    for op, saved, fn in cases:
        want = la.la_workspace_bytes(op, B, H, N, D, M, tdt, saved=saved)
        assert want == la.la_workspace_bytes(op, B, H, N, D, M, tdt, saved=saved, num_sms=sms)
        peak = _peak_of(fn)
        # the pool hands out whole allocation granules: the peak is the reported
        # bytes rounded up to at most 2 MiB per allocation, never less
        assert want <= peak <= want + 4 * (2 << 20), (op, saved, want, peak)
    assert _peak_of(fwd) >= 0
    la.la_check_device_status()


def test_noncausal_backward_bytes():
    # fp32 D = M = 64 on the tensor cores: the forward's state partials (4 spans per head
    # at two CTAs per SM) plus the query side's (R | r) partials, also two CTAs per SM: 32
    # chunks per head cut into 4 spans of 8 chunks (256 CTAs, one wave of 304 slots: the
    # fewest waves x chunks, fewest spans on a tie with 8 spans of 4), 64 heads
    up = lambda x: (x + 255) // 256 * 256
    W = 64 * 64 + 64
    assert _ws("la_backward_noncausal", 8, 8, 4096, 64, 64, F32) == up(4 * 64 * 4 * W) + 4 * 64 * 4 * W
    # other shapes on the CUDA cores: state and (R | r) partials and totals
    assert _ws("la_backward_noncausal", 1, 2, 1000, 32, 64, BF16) > 0
