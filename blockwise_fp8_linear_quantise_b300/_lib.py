"""ctypes declarations of the C ABI in include/bfp8.h (libbfp8.so)."""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbfp8.so")

c_i64 = ctypes.c_int64
c_p = ctypes.c_void_p
c_sz = ctypes.c_size_t
c_int = ctypes.c_int


class WJob(ctypes.Structure):
    """bfp8_w_job: one weight of bfp8_quantize_w_128x128_batch."""
    _fields_ = [("w", c_p), ("n", c_i64), ("k", c_i64), ("q", c_p), ("qT", c_p), ("s", c_p)]


# name -> (restype, argtypes), in the order the header declares them
SIGNATURES = {
    "bfp8_quantize_act_1x128": (c_int, [c_p, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p]),
    "bfp8_quantize_w_128x128": (c_int, [c_p, c_i64, c_i64, c_p, c_p, c_p, c_p]),
    "bfp8_quantize_act_1x128_ex": (c_int, [c_p, c_i64, c_i64, c_p, c_p, c_p, c_p, c_int, c_p]),
    "bfp8_quantize_w_128x128_ex": (c_int, [c_p, c_i64, c_i64, c_p, c_p, c_p, c_int, c_p]),
    "bfp8_quantize_w_128x128_batch": (c_int, [ctypes.POINTER(WJob), c_int, c_int, c_p]),
    "bfp8_swiglu_quantize_1x128": (c_int, [c_p, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p, c_int, c_p]),
    "bfp8_quantize_mx_1x32": (c_int, [c_p, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p]),
    "bfp8_mx_gemm": (c_int, [c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p]),
    "bfp8_fp8_block_gemm": (c_int, [c_int, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "bfp8_gemm_workspace_bytes": (c_sz, [c_int, c_i64, c_i64, c_i64]),
    "bfp8_fp8_block_gemm_accumulate": (c_int, [c_int, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_sz, c_p]),
    "bfp8_fp8_block_gemm_noalloc": (c_int, [c_int, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p]),
    "bfp8_linear_fwd": (c_int, [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "bfp8_linear_fwd_workspace_bytes": (c_sz, [c_i64, c_i64, c_i64]),
    "bfp8_linear_bwd": (c_int, [c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_sz, c_p]),
    "bfp8_linear_bwd_workspace_bytes": (c_sz, [c_i64, c_i64, c_i64]),
    "bfp8_linear_fwd_prequantised": (c_int, [c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p, c_sz, c_int,
                                             c_p]),
    "bfp8_linear_fwd_ex": (c_int, [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_int, c_p]),
    "bfp8_linear_bwd_ex": (c_int, [c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_sz, c_int, c_p]),
    "bfp8_linear_bwd_main_grad": (c_int, [c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_sz, c_int,
                                          c_p]),
    "bfp8_sync_status": (c_int, [c_p]),
    "bfp8_set_wait_limit_ns": (c_int, [ctypes.c_uint64]),
    "bfp8_set_gemm_kernel": (c_int, [c_int]),
    "bfp8_set_gemm_splits": (c_int, [c_int]),
    "bfp8_launch_count": (ctypes.c_uint64, []),
    "bfp8_test_stall_next_launch": (c_int, []),
    "bfp8_status_string": (ctypes.c_char_p, [c_int]),
}

STATUS = {0: "BFP8_OK", 1: "BFP8_EINVAL", 2: "BFP8_EALIGN", 3: "BFP8_EUNSUPPORTED", 4: "BFP8_ECUDA",
          5: "BFP8_ETIMEOUT", 6: "BFP8_EWORKSPACE"}
STATUS_CODE = {v: k for k, v in STATUS.items()}

_lib = None


def load():
    """Load libbfp8.so once and declare every entry point; raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc for sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
