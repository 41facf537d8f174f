"""ctypes loader for liblinattn.so (the C ABI declared in include/linattn.h).

There is no fallback: if the library is missing or fails to load, importing
this module raises, so nothing can silently run on the CPU or through torch.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "liblinattn.so")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(5)
LA_DTYPE_F32, LA_DTYPE_BF16 = 0, 1
LA_SAVED_OUT, LA_SAVED_DEN, LA_SAVED_CKPT = 1, 2, 4
SIZE_MAX = ctypes.c_size_t(-1).value

# (name, argtypes) of every exported entry point.
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "la_forward_causal": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _F, _F, _F, _P],
    "la_backward_causal": [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _P],
    "la_causal_ckpt_floats": [_I, _I, _I, _I, _I],
    "la_forward_noncausal": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
    "la_forward_noncausal_noalloc": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
    "la_backward_noncausal": [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
    "la_decode_step": [_P, _P, _P, _F, _F, _F, _I, _I, _I, _I, _I, _P],
    "la_workspace_bytes": [ctypes.c_char_p, _I, _I, _I, _I, _I, _I, ctypes.c_uint, _I],
    "la_scratch_peak_bytes": [_I],
    "la_forward_poly2": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P],
    "la_forward_retention": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _F, _P],
    "la_retention_decode_step": [_P, _P, _P, _F, _F, _F, _F, _I, _I, _I, _I, _I, _P],
    "la_softmax_decode_step": [_P, _P, _P, _P, _P, _I, _I, _F, _I, _I, _I, _I, _I, _P],
    "la_debug_withhold_publication": [_I, ctypes.c_uint],
    "la_check_device_status": [_P],
    "la_selftest_expired_waits": [_P],
    "la_status_string": [_I],
    "la_last_error_message": [],
    "la_kernel_launch_count": [],
}
_RESTYPES = {"la_status_string": ctypes.c_char_p, "la_last_error_message": ctypes.c_char_p,
             "la_causal_ckpt_floats": ctypes.c_size_t, "la_workspace_bytes": ctypes.c_size_t,
             "la_scratch_peak_bytes": ctypes.c_size_t,
             "la_kernel_launch_count": ctypes.c_uint64}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(needs nvcc); the library has no CPU fallback")
    lib = ctypes.CDLL(path)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _RESTYPES.get(name, ctypes.c_int)
    return lib


lib = load()
