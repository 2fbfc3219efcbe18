"""The C-ABI library loads without a GPU, exports every entry point that
include/bfp8.h declares, and rejects bad arguments on the host (these checks
run before any device is touched)."""

import ctypes
import os
import re

import pytest

from conftest import ROOT
from blockwise_fp8_linear_quantise_b300 import _lib

HEADER = os.path.join(ROOT, "include", "bfp8.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bfp8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("bfp8_quantize_act_1x128", "bfp8_quantize_w_128x128", "bfp8_fp8_block_gemm",
                     "bfp8_linear_fwd", "bfp8_linear_bwd", "bfp8_sync_status", "bfp8_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"


def test_launch_count_starts_without_gpu_work():
    # argument errors launch nothing, so the counter does not move
    lib = _lib.load()
    before = lib.bfp8_launch_count()
    assert lib.bfp8_quantize_act_1x128(None, 128, 128, FAKE, FAKE, None, None, None) != 0
    assert lib.bfp8_launch_count() == before


def test_status_strings():
    lib = _lib.load()
    for code in range(7):
        assert lib.bfp8_status_string(code)
    assert b"unknown" in lib.bfp8_status_string(99)


EINVAL, EALIGN, EWORKSPACE = 1, 2, 6
FAKE = 0x10000  # never dereferenced: validation fails first
MIS = 0x10001


@pytest.mark.parametrize("M,K", [(0, 128), (128, 0), (100, 128), (128, 130), (-128, 128)])
def test_quantize_rejects_bad_dims(M, K):
    lib = _lib.load()
    assert lib.bfp8_quantize_act_1x128(FAKE, M, K, FAKE, FAKE, None, None, None) == EINVAL
    assert lib.bfp8_quantize_w_128x128(FAKE, M, K, FAKE, None, FAKE, None) == EINVAL


def test_quantize_rejects_nulls_and_misalignment():
    lib = _lib.load()
    assert lib.bfp8_quantize_act_1x128(None, 128, 128, FAKE, FAKE, None, None, None) == EINVAL
    assert lib.bfp8_quantize_act_1x128(FAKE, 128, 128, None, None, None, None, None) == EINVAL
    assert lib.bfp8_quantize_act_1x128(FAKE, 128, 128, FAKE, None, None, None, None) == EINVAL
    assert lib.bfp8_quantize_act_1x128(FAKE, 128, 128, None, None, FAKE, None, None) == EINVAL
    assert lib.bfp8_quantize_act_1x128(MIS, 128, 128, FAKE, FAKE, None, None, None) == EALIGN
    assert lib.bfp8_quantize_act_1x128(FAKE, 128, 128, FAKE, MIS, None, None, None) == EALIGN
    assert lib.bfp8_quantize_w_128x128(FAKE, 128, 128, FAKE, FAKE, None, None) == EINVAL
    assert lib.bfp8_quantize_w_128x128(FAKE, 128, 128, None, None, FAKE, None) == EINVAL
    assert lib.bfp8_quantize_w_128x128(FAKE, 128, 128, FAKE, MIS, FAKE, None) == EALIGN


def test_swiglu_quantize_rejects_bad_arguments():
    f = _lib.load().bfp8_swiglu_quantize_1x128
    assert f(None, 128, 128, None, FAKE, FAKE, None, None, 0, None) == EINVAL
    assert f(FAKE, 128, 128, FAKE, None, None, None, None, 0, None) == EINVAL  # no codes requested
    assert f(FAKE, 128, 128, None, FAKE, None, None, None, 0, None) == EINVAL  # q without s
    assert f(FAKE, 128, 128, None, None, None, FAKE, None, 0, None) == EINVAL  # qT without sT
    assert f(FAKE, 128, 100, None, FAKE, FAKE, None, None, 0, None) == EINVAL
    assert f(FAKE, 0, 128, None, FAKE, FAKE, None, None, 0, None) == EINVAL
    assert f(FAKE, 128, 128, None, FAKE, FAKE, None, None, 5, None) == EINVAL
    assert f(MIS, 128, 128, None, FAKE, FAKE, None, None, 0, None) == EALIGN
    assert f(FAKE, 128, 128, MIS, FAKE, FAKE, None, None, 0, None) == EALIGN
    assert f(FAKE, 128, 128, None, FAKE, FAKE, MIS, FAKE, 0, None) == EALIGN


def test_gemm_rejects_bad_arguments():
    lib = _lib.load()
    g = lib.bfp8_fp8_block_gemm
    assert g(3, FAKE, FAKE, FAKE, FAKE, 128, 128, 128, FAKE, None, None, None, 0, None) == EINVAL
    assert g(0, None, FAKE, FAKE, FAKE, 128, 128, 128, FAKE, None, None, None, 0, None) == EINVAL
    assert g(0, FAKE, FAKE, FAKE, FAKE, 128, 192, 128, FAKE, None, None, None, 0, None) == EINVAL
    assert g(0, FAKE, FAKE, FAKE, FAKE, 128, 128, 128, FAKE, FAKE, None, None, 0, None) == EINVAL
    assert g(0, MIS, FAKE, FAKE, FAKE, 128, 128, 128, FAKE, None, None, None, 0, None) == EALIGN
    assert g(2, FAKE, FAKE, FAKE, FAKE, 128, 128, 128, MIS, None, None, None, 0, None) == EALIGN


def test_linear_rejects_bad_arguments():
    lib = _lib.load()
    assert lib.bfp8_linear_fwd(None, FAKE, 128, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == EINVAL
    assert lib.bfp8_linear_fwd(FAKE, FAKE, 128, 128, 100, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == EINVAL
    assert lib.bfp8_linear_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 0, 128, FAKE, FAKE, FAKE, 1 << 20, None) == EINVAL
    assert lib.bfp8_set_gemm_splits(-1) == EINVAL


def test_workspace_sizes_cover_the_intermediates():
    lib = _lib.load()
    M, N, K = 8192, 2048, 6144
    fwd = lib.bfp8_linear_fwd_workspace_bytes(M, N, K)
    assert fwd >= N * K + M * K + (K // 128) * M * 4       # Wq + Xq + sX
    bwd = lib.bfp8_linear_bwd_workspace_bytes(M, N, K)
    assert bwd >= 2 * M * N + (N // 128) * M * 4 + (M // 128) * N * 4  # dYq + dYqT + scales
    assert lib.bfp8_linear_fwd_workspace_bytes(M, N, 100) == 0
    assert lib.bfp8_gemm_workspace_bytes(0, 100, 128, 128) == 0


def test_weight_batch_rejects_bad_jobs():
    from blockwise_fp8_linear_quantise_b300._lib import WJob
    lib = _lib.load()
    f = lib.bfp8_quantize_w_128x128_batch
    good = lambda: WJob(FAKE, 256, 128, FAKE, FAKE, FAKE)
    jobs = (WJob * 3)(good(), good(), good())
    assert f(None, 1, 0, None) == EINVAL
    assert f(jobs, 0, 0, None) == EINVAL
    assert f(jobs, 3, 7, None) == EINVAL                      # unknown scale mode
    for bad, want in ((WJob(None, 256, 128, FAKE, FAKE, FAKE), EINVAL),   # no weight
                      (WJob(FAKE, 256, 128, FAKE, FAKE, None), EINVAL),   # no scales
                      (WJob(FAKE, 256, 128, None, FAKE, FAKE), EINVAL),   # outputs differ from job 0's
                      (WJob(FAKE, 200, 128, FAKE, FAKE, FAKE), EINVAL),   # not a multiple of 128
                      (WJob(MIS, 256, 128, FAKE, FAKE, FAKE), EALIGN),
                      (WJob(FAKE, 256, 128, FAKE, MIS, FAKE), EALIGN)):
        jobs[2] = bad
        assert f(jobs, 3, 0, None) == want
    assert f((WJob * 1)(WJob(FAKE, 256, 128, None, None, FAKE)), 1, 0, None) == EINVAL  # no output at all
