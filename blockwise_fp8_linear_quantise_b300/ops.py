"""torch-facing wrappers of the C ABI (argument marshalling only).

Every function checks dtypes/shapes of the torch tensors it is given,
allocates missing outputs with torch on the input's device, passes raw
pointers and the current CUDA stream to libbfp8.so and raises
``BFP8Error`` on a non-OK status.  All arithmetic happens in the CUDA
kernels behind the ABI.

Layouts are those of include/bfp8.h: E4M3 codes are torch.uint8 tensors,
scales are float32, activation scales are group-major ([K/128, M] for a
[M, K] tensor quantised along K).
"""

import torch

from . import _lib

FPROP, DGRAD, WGRAD = 0, 1, 2


class BFP8Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        lib = _lib.load()
        super().__init__(f"{what}: {_lib.STATUS.get(status, status)} ({lib.bfp8_status_string(status).decode()})")


def _check(status, what):
    if status != 0:
        raise BFP8Error(status, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")
    return t


def _out(t, dtype, shape, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _need(t, dtype, shape, name)


SCALE_MODES = {"amax448": 0, "pow2": 1, "mul_recip": 2}


def _scale_mode(scale_mode):
    try:
        return SCALE_MODES[scale_mode]
    except KeyError:
        raise ValueError(f"unknown scale_mode {scale_mode!r}") from None


def quantize_act_1x128(x, rows=True, tokens=False, q=None, s=None, qT=None, sT=None, stream=None,
                       scale_mode="amax448"):
    """Quantise bf16 x [M, K] in 1x128 groups.

    rows   -> q [M, K] uint8 (groups along K), s [K/128, M] float32
    tokens -> qT [K, M] uint8 (groups of 128 tokens per column), sT [M/128, K]
    scale_mode "amax448" (s = amax/448, codes of x/s), "pow2" (smallest power of two >= amax/448) or
    "mul_recip" (s = amax/448, codes of x * fp32(448/amax)).
    Returns (q, s, qT, sT) with None for outputs not requested.
    """
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    if rows:
        q = _out(q, torch.uint8, (M, K), x.device, "q")
        s = _out(s, torch.float32, (K // 128, M), x.device, "s")
    else:
        q = s = None
    if tokens:
        qT = _out(qT, torch.uint8, (K, M), x.device, "qT")
        sT = _out(sT, torch.float32, (M // 128, K), x.device, "sT")
    else:
        qT = sT = None
    lib = _lib.load()
    _check(lib.bfp8_quantize_act_1x128_ex(_ptr(x), M, K, _ptr(q), _ptr(s), _ptr(qT), _ptr(sT),
                                          _scale_mode(scale_mode), _stream(stream)),
           "quantize_act_1x128")
    return q, s, qT, sT


def swiglu_quantize_1x128(gu, rows=True, tokens=True, want_h=False, h=None, q=None, s=None, qT=None, sT=None,
                          stream=None, scale_mode="amax448"):
    """The down projection's input from the gate+up output gu [M, 2F] (gate in
    columns 0..F-1, up in F..2F-1): h = bf16(SiLU(g) * u), quantised in 1x128
    groups as quantize_act_1x128(h, rows, tokens) does, in one pass.

    Returns (h or None, q, s, qT, sT); h [M, F] bf16 is written only when
    want_h (or h) is given.
    """
    M, F2 = gu.shape
    _need(gu, torch.bfloat16, (M, F2), "gu")
    if F2 % 2:
        raise ValueError("gu must have an even number of columns")
    F = F2 // 2
    h = _out(h, torch.bfloat16, (M, F), gu.device, "h") if (want_h or h is not None) else None
    if rows:
        q = _out(q, torch.uint8, (M, F), gu.device, "q")
        s = _out(s, torch.float32, (F // 128, M), gu.device, "s")
    else:
        q = s = None
    if tokens:
        qT = _out(qT, torch.uint8, (F, M), gu.device, "qT")
        sT = _out(sT, torch.float32, (M // 128, F), gu.device, "sT")
    else:
        qT = sT = None
    lib = _lib.load()
    _check(lib.bfp8_swiglu_quantize_1x128(_ptr(gu), M, F, _ptr(h), _ptr(q), _ptr(s), _ptr(qT), _ptr(sT),
                                          _scale_mode(scale_mode), _stream(stream)),
           "swiglu_quantize_1x128")
    return h, q, s, qT, sT


def quantize_w_128x128(w, want_q=True, want_qT=True, q=None, qT=None, s=None, stream=None, scale_mode="amax448"):
    """Quantise bf16 w [N, K] in 128x128 blocks -> (q [N, K], qT [K, N], s [N/128, K/128]).

    scale_mode as for quantize_act_1x128."""
    N, K = w.shape
    _need(w, torch.bfloat16, (N, K), "w")
    q = _out(q, torch.uint8, (N, K), w.device, "q") if want_q else None
    qT = _out(qT, torch.uint8, (K, N), w.device, "qT") if want_qT else None
    s = _out(s, torch.float32, (N // 128, K // 128), w.device, "s")
    lib = _lib.load()
    _check(lib.bfp8_quantize_w_128x128_ex(_ptr(w), N, K, _ptr(q), _ptr(qT), _ptr(s), _scale_mode(scale_mode),
                                          _stream(stream)),
           "quantize_w_128x128")
    return q, qT, s


def quantize_w_batch(ws, want_q=True, want_qT=True, outs=None, stream=None, scale_mode="amax448"):
    """Quantise several bf16 weights (each [N, K]) in 128x128 blocks with one
    launch per four weights -> [(q, qT, s), ...], each as quantize_w_128x128
    returns it.  outs: optional [(q, qT, s), ...] to write into."""
    lib = _lib.load()
    res = []
    jobs = (_lib.WJob * len(ws))()
    for i, w in enumerate(ws):
        N, K = w.shape
        _need(w, torch.bfloat16, (N, K), "w")
        oq, oqT, os_ = outs[i] if outs is not None else (None, None, None)
        q = _out(oq, torch.uint8, (N, K), w.device, "q") if want_q else None
        qT = _out(oqT, torch.uint8, (K, N), w.device, "qT") if want_qT else None
        s = _out(os_, torch.float32, (N // 128, K // 128), w.device, "s")
        jobs[i] = _lib.WJob(_ptr(w), N, K, _ptr(q), _ptr(qT), _ptr(s))
        res.append((q, qT, s))
    _check(lib.bfp8_quantize_w_128x128_batch(jobs, len(ws), _scale_mode(scale_mode), _stream(stream)),
           "quantize_w_batch")
    return res


def quantize_mx_1x32(x, rows=True, tokens=False, q=None, s=None, qT=None, sT=None, stream=None):
    """MXFP8 1x32 quantisation of bf16 x [M, K] (power-of-two scales per 32 values).

    rows   -> q [M, K] uint8 (groups of 32 along K), s [K/32, M] float32
    tokens -> qT [K, M] uint8 (groups of 32 rows per column), sT [M/32, K]
    Returns (q, s, qT, sT) with None for outputs not requested.
    """
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    if rows:
        q = _out(q, torch.uint8, (M, K), x.device, "q")
        s = _out(s, torch.float32, (K // 32, M), x.device, "s")
    else:
        q = s = None
    if tokens:
        qT = _out(qT, torch.uint8, (K, M), x.device, "qT")
        sT = _out(sT, torch.float32, (M // 32, K), x.device, "sT")
    else:
        qT = sT = None
    _check(_lib.load().bfp8_quantize_mx_1x32(_ptr(x), M, K, _ptr(q), _ptr(s), _ptr(qT), _ptr(sT), _stream(stream)),
           "quantize_mx_1x32")
    return q, s, qT, sT


def mx_gemm(A, sa, B, sb, C=None, stream=None):
    """C [M, N] bf16 = A . B^T with 1x32 scales along K for both operands (A [M, K], sa [K/32, M], B [N, K],
    sb [K/32, N])."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, torch.uint8, (M, K), "A")
    _need(B, torch.uint8, (N, K), "B")
    _need(sa, torch.float32, (K // 32, M), "sa")
    _need(sb, torch.float32, (K // 32, N), "sb")
    C = _out(C, torch.bfloat16, (M, N), A.device, "C")
    _check(_lib.load().bfp8_mx_gemm(_ptr(A), _ptr(sa), _ptr(B), _ptr(sb), M, N, K, _ptr(C), _stream(stream)),
           "mx_gemm")
    return C


def gemm_workspace_bytes(layout, M, N, K):
    return int(_lib.load().bfp8_gemm_workspace_bytes(layout, M, N, K))


def fp8_block_gemm(layout, A, sa, B, sb, C=None, fused_quant=False, Cq=None, sCq=None, workspace=None, stream=None):
    """Block-scaled GEMM C [M, N] = sum_kb (A . B^T)_kb * sa * sb, bf16 out.

    A uint8 [M, K], B uint8 [N, K], sa float32 [K/128, M]; sb per layout:
    FPROP [N/128, K/128], DGRAD [K/128, N/128], WGRAD [K/128, N].
    With fused_quant also returns the E4M3 codes of C (groups along N).
    Returns C or (C, Cq, sCq).
    """
    M, K = A.shape
    N = B.shape[0]
    _need(A, torch.uint8, (M, K), "A")
    _need(B, torch.uint8, (N, K), "B")
    _need(sa, torch.float32, (K // 128, M), "sa")
    sb_shape = {FPROP: (N // 128, K // 128), DGRAD: (K // 128, N // 128), WGRAD: (K // 128, N)}[layout]
    _need(sb, torch.float32, sb_shape, "sb")
    C = _out(C, torch.bfloat16, (M, N), A.device, "C")
    if fused_quant:
        Cq = _out(Cq, torch.uint8, (M, N), A.device, "Cq")
        sCq = _out(sCq, torch.float32, (N // 128, M), A.device, "sCq")
    else:
        Cq = sCq = None
    need = gemm_workspace_bytes(layout, M, N, K)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = _lib.load()
    _check(lib.bfp8_fp8_block_gemm(layout, _ptr(A), _ptr(sa), _ptr(B), _ptr(sb), M, N, K, _ptr(C), _ptr(Cq),
                                   _ptr(sCq), _ptr(workspace), ws_bytes, _stream(stream)), "fp8_block_gemm")
    return (C, Cq, sCq) if fused_quant else C


def fp8_block_gemm_accumulate(layout, A, sa, B, sb, C_f32, workspace=None, stream=None):
    """C_f32 [M, N] (fp32, updated in place) += the block-scaled product of
    fp8_block_gemm's operands.  Returns C_f32."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, torch.uint8, (M, K), "A")
    _need(B, torch.uint8, (N, K), "B")
    _need(sa, torch.float32, (K // 128, M), "sa")
    sb_shape = {FPROP: (N // 128, K // 128), DGRAD: (K // 128, N // 128), WGRAD: (K // 128, N)}[layout]
    _need(sb, torch.float32, sb_shape, "sb")
    _need(C_f32, torch.float32, (M, N), "C_f32")
    ws_n = gemm_workspace_bytes(layout, M, N, K)
    if workspace is None:
        workspace = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=A.device)
    lib = _lib.load()
    _check(lib.bfp8_fp8_block_gemm_accumulate(layout, _ptr(A), _ptr(sa), _ptr(B), _ptr(sb), M, N, K, _ptr(C_f32),
                                              _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp8_block_gemm_accumulate")
    return C_f32


def linear_fwd_workspace_bytes(M, N, K):
    return int(_lib.load().bfp8_linear_fwd_workspace_bytes(M, N, K))


def linear_bwd_workspace_bytes(M, N, K):
    return int(_lib.load().bfp8_linear_bwd_workspace_bytes(M, N, K))


def linear_fwd(X, W, Y=None, saved=None, workspace=None, stream=None, scale_mode="amax448"):
    """Y = X . W^T through the fused forward.  Returns (Y, saved) where saved
    holds WqT, sW, XqT, sXT for linear_bwd.  scale_mode as for
    quantize_act_1x128."""
    M, K = X.shape
    N = W.shape[0]
    _need(X, torch.bfloat16, (M, K), "X")
    _need(W, torch.bfloat16, (N, K), "W")
    dev = X.device
    Y = _out(Y, torch.bfloat16, (M, N), dev, "Y")
    if saved is None:
        saved = dict(WqT=torch.empty((K, N), dtype=torch.uint8, device=dev),
                     sW=torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev),
                     XqT=torch.empty((K, M), dtype=torch.uint8, device=dev),
                     sXT=torch.empty((M // 128, K), dtype=torch.float32, device=dev))
    if workspace is None:
        workspace = torch.empty(linear_fwd_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    lib = _lib.load()
    _check(lib.bfp8_linear_fwd_ex(_ptr(X), _ptr(W), M, N, K, _ptr(Y), _ptr(saved["WqT"]), _ptr(saved["sW"]),
                                  _ptr(saved["XqT"]), _ptr(saved["sXT"]), _ptr(workspace), workspace.numel(),
                                  _scale_mode(scale_mode), _stream(stream)), "linear_fwd")
    return Y, saved


def linear_fwd_prequantised(X, Wq, sW, WqT=None, Y=None, saved=None, workspace=None, stream=None,
                            scale_mode="amax448"):
    """Y = X . W^T with W's codes Wq [N, K] and scales sW [N/128, K/128]
    quantised earlier (quantize_w_128x128), e.g. once per optimizer step.
    Returns (Y, saved) like linear_fwd; saved takes WqT (when given) and sW
    for linear_bwd."""
    M, K = X.shape
    N = Wq.shape[0]
    _need(X, torch.bfloat16, (M, K), "X")
    _need(Wq, torch.uint8, (N, K), "Wq")
    _need(sW, torch.float32, (N // 128, K // 128), "sW")
    dev = X.device
    Y = _out(Y, torch.bfloat16, (M, N), dev, "Y")
    if saved is None:
        saved = dict(XqT=torch.empty((K, M), dtype=torch.uint8, device=dev),
                     sXT=torch.empty((M // 128, K), dtype=torch.float32, device=dev))
    saved["sW"] = sW
    if WqT is not None:
        saved["WqT"] = WqT
    if workspace is None:
        workspace = torch.empty(linear_fwd_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    lib = _lib.load()
    _check(lib.bfp8_linear_fwd_prequantised(_ptr(X), _ptr(Wq), _ptr(sW), M, N, K, _ptr(Y), _ptr(saved["XqT"]),
                                            _ptr(saved["sXT"]), _ptr(workspace), workspace.numel(),
                                            _scale_mode(scale_mode), _stream(stream)), "linear_fwd_prequantised")
    return Y, saved


def linear_bwd(dY, saved, dX=None, dW=None, workspace=None, stream=None, scale_mode="amax448", dW_main=None):
    """(dX, dW) for the layer whose forward produced ``saved``; scale_mode
    applies to the quantisation of dY.  With dW_main (fp32 [N, K]) the weight
    gradient is added into it instead and (dX, dW_main) is returned."""
    M, N = dY.shape
    K = saved["WqT"].shape[0]
    _need(dY, torch.bfloat16, (M, N), "dY")
    _need(saved["WqT"], torch.uint8, (K, N), "WqT")
    _need(saved["sW"], torch.float32, (N // 128, K // 128), "sW")
    _need(saved["XqT"], torch.uint8, (K, M), "XqT")
    _need(saved["sXT"], torch.float32, (M // 128, K), "sXT")
    dev = dY.device
    dX = _out(dX, torch.bfloat16, (M, K), dev, "dX")
    if workspace is None:
        workspace = torch.empty(linear_bwd_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    lib = _lib.load()
    if dW_main is not None:
        _need(dW_main, torch.float32, (N, K), "dW_main")
        _check(lib.bfp8_linear_bwd_main_grad(_ptr(dY), _ptr(saved["WqT"]), _ptr(saved["sW"]), _ptr(saved["XqT"]),
                                             _ptr(saved["sXT"]), M, N, K, _ptr(dX), _ptr(dW_main), _ptr(workspace),
                                             workspace.numel(), _scale_mode(scale_mode), _stream(stream)),
               "linear_bwd_main_grad")
        return dX, dW_main
    dW = _out(dW, torch.bfloat16, (N, K), dev, "dW")
    _check(lib.bfp8_linear_bwd_ex(_ptr(dY), _ptr(saved["WqT"]), _ptr(saved["sW"]), _ptr(saved["XqT"]),
                                  _ptr(saved["sXT"]), M, N, K, _ptr(dX), _ptr(dW), _ptr(workspace),
                                  workspace.numel(), _scale_mode(scale_mode), _stream(stream)), "linear_bwd")
    return dX, dW


def sync_status(stream=None):
    """Synchronise the stream and return the device-side status code (0 = ok)."""
    return int(_lib.load().bfp8_sync_status(_stream(stream)))


def set_wait_limit_ns(ns):
    _check(_lib.load().bfp8_set_wait_limit_ns(int(ns)), "set_wait_limit_ns")


def set_gemm_kernel(kind):
    """0: CTA-pair 256x256 tiles for FPROP/DGRAD where the shape allows (default); 1: single-CTA tiles only;
    2: CTA pairs for WGRAD as well."""
    _check(_lib.load().bfp8_set_gemm_kernel(int(kind)), "set_gemm_kernel")


def set_gemm_splits(splits):
    _check(_lib.load().bfp8_set_gemm_splits(int(splits)), "set_gemm_splits")


def launch_count():
    """Kernels the library has launched in this process so far."""
    return int(_lib.load().bfp8_launch_count())


def test_stall_next_launch():
    """Test hook: the next quantiser or GEMM launch makes one bounded wait that nothing satisfies (it expires
    after the wait limit, and sync_status() then reports BFP8_ETIMEOUT)."""
    _check(_lib.load().bfp8_test_stall_next_launch(), "test_stall_next_launch")
