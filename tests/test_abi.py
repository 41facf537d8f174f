"""Host-side checks of the C ABI: the library loads, exports every entry point
declared in include/linattn.h, and rejects bad arguments before touching CUDA.
No call here reaches a kernel (every case fails validation first)."""
import ctypes
import os
import re

import pytest

from linear_attention_02_gb300 import _native

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "linattn.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_paths():
    names = _declared()
    for n in ("la_forward_causal", "la_backward_causal", "la_forward_noncausal", "la_decode_step"):
        assert n in names


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(_native.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(_native.SIGNATURES)


def test_status_strings():
    lib = _native.lib
    assert lib.la_status_string(0) == b"LA_OK"
    assert lib.la_status_string(4) == b"LA_ERR_TIMEOUT"
    assert lib.la_status_string(99) == b"LA_ERR_UNKNOWN"


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("D,M,status", [(48, 64, _native.LA_ERR_UNSUPPORTED),
                                        (64, 16, _native.LA_ERR_UNSUPPORTED),
                                        (256, 64, _native.LA_ERR_UNSUPPORTED)])
def test_unsupported_head_sizes(D, M, status):
    lib = _native.lib
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, D, M, 0, None, None, None, None, None, None,
                                 None) == status
    assert b"head sizes" in lib.la_last_error_message()


def test_invalid_arguments():
    lib = _native.lib
    E = _native.LA_ERR_INVALID_ARG
    # null and misaligned pointers
    assert lib.la_forward_causal(None, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64, 0, None, None, None, None, None, None,
                                 None) == E
    assert b"Q is NULL" in lib.la_last_error_message()
    assert lib.la_forward_causal(FAKE, FAKE + 4, FAKE, FAKE, 1, 1, 8, 64, 64, 0, None, None, None,
                                 None, None, None, None) == E
    assert b"K is not 16-byte aligned" in lib.la_last_error_message()
    # negative sizes, unpaired states, bad dtype
    assert lib.la_forward_noncausal(FAKE, FAKE, FAKE, FAKE, 1, -1, 8, 64, 64, 0, None) == E
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64, 0, FAKE, None, None, None, None, None,
                                 None) == E
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64, 0, None, None, None, FAKE, None, None,
                                 None) == E
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64, 7, None, None, None, None, None, None,
                                 None) == _native.LA_ERR_UNSUPPORTED
    assert lib.la_backward_causal(FAKE, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, 1, 1, 8, 64, 64,
                                  1, None, None, None) == E
    assert b"dK is NULL" in lib.la_last_error_message()
    # the optional normaliser must be aligned like every other buffer
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64, 1, None, None, None, None,
                                 FAKE + 4, None, None) == E
    assert b"Den is not 16-byte aligned" in lib.la_last_error_message()
    assert lib.la_backward_causal(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64,
                                  1, FAKE + 4, None, None) == E
    assert b"Den is not 16-byte aligned" in lib.la_last_error_message()
    assert lib.la_backward_causal(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64,
                                  1, None, FAKE + 8, None) == E
    assert b"Ckpt is not 16-byte aligned" in lib.la_last_error_message()
    # checkpoint size: B H ceil(ceil(N / 128) / 8) (D M + D) words
    assert lib.la_causal_ckpt_floats(4, 16, 8192, 64, 64) == 4 * 16 * 8 * (64 * 64 + 64)
    assert lib.la_causal_ckpt_floats(1, 1, 1025 * 1, 64, 64) == 2 * (64 * 64 + 64)
    assert lib.la_causal_ckpt_floats(1, 1, 0, 64, 64) == 0
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE + 8, FAKE, 2, 2, 64, 64, 1, None) == E
    # too large
    assert lib.la_forward_noncausal(FAKE, FAKE, FAKE, FAKE, 1 << 20, 1 << 10, 1 << 20, 64, 64, 0,
                                    None) == E


def test_empty_calls_succeed_without_a_device():
    lib = _native.lib
    # B*H*N == 0 with no state requested: nothing to do, no CUDA call is made
    assert lib.la_backward_causal(None, None, None, None, None, None, None, None, 2, 3, 0, 64, 64,
                                  1, None, None, None) == _native.LA_OK
    assert lib.la_forward_noncausal(None, None, None, None, 0, 4, 100, 32, 32, 0, None) == _native.LA_OK
    assert lib.la_decode_step(None, None, None, None, None, None, 0, 16, 64, 64, 1, None) == _native.LA_OK
