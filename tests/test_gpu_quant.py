"""GPU quantisers vs the CPU oracle: E4M3 codes and fp32 scales bit-exact, in
every scale mode (amax/448, power-of-two, and the reciprocal multiply)."""

import numpy as np
import pytest
import torch

from gpu_helpers import (assert_codes_equal, assert_scales_equal, bf16_input, dev, np32, u8, to_gpu)
from oracle import quant
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu


def check_act(x_bf16, scale_mode="amax448"):
    x = x_bf16.to(dev())
    q, s, qT, sT = ops.quantize_act_1x128(x, rows=True, tokens=True, scale_mode=scale_mode)
    torch.cuda.synchronize()
    assert ops.sync_status() == 0
    xn = np32(x_bf16)
    oq, os_ = quant.quantize_act_1x128(xn, scale_mode=scale_mode)
    oqT, osT = quant.quantize_act_tokens_1x128(xn, scale_mode=scale_mode)
    assert_codes_equal(u8(q), oq, "q")
    assert_scales_equal(s.cpu().numpy(), os_, "s")
    assert_codes_equal(u8(qT), oqT, "qT")
    assert_scales_equal(sT.cpu().numpy(), osT, "sT")
    # single-output variants give the same bytes
    q2, s2, _, _ = ops.quantize_act_1x128(x, rows=True, tokens=False, scale_mode=scale_mode)
    _, _, qT2, sT2 = ops.quantize_act_1x128(x, rows=False, tokens=True, scale_mode=scale_mode)
    assert torch.equal(q2, q) and torch.equal(s2, s) and torch.equal(qT2, qT) and torch.equal(sT2, sT)


def check_w(w_bf16, scale_mode="amax448"):
    w = w_bf16.to(dev())
    q, qT, s = ops.quantize_w_128x128(w, scale_mode=scale_mode)
    assert ops.sync_status() == 0
    oq, oqT, os_ = quant.quantize_w_128x128(np32(w_bf16), scale_mode=scale_mode)
    assert_codes_equal(u8(q), oq, "Wq")
    assert_codes_equal(u8(qT), oqT, "WqT")
    assert_scales_equal(s.cpu().numpy(), os_, "sW")
    q1, _, s1 = ops.quantize_w_128x128(w, want_qT=False, scale_mode=scale_mode)
    _, qT1, _ = ops.quantize_w_128x128(w, want_q=False, scale_mode=scale_mode)
    assert torch.equal(q1, q) and torch.equal(qT1, qT) and torch.equal(s1, s)


def test_tiny_config():
    check_act(bf16_input("tiny", "x"))
    check_w(bf16_input("tiny", "w"))


@pytest.mark.parametrize("M,K", [(128, 128), (384, 640), (1152, 256)])
def test_multi_tile_shapes(M, K):
    rng = np.random.default_rng(M * 7 + K)
    x = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32) * np.exp2(rng.integers(-20, 20, (M, 1))))
    check_act(x)
    check_w(x)


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
def test_edge_values(scale_mode):
    # zeros (scale 1), signed zeros, subnormal-scale groups, huge groups, ties
    M, K = 256, 384
    x = np.zeros((M, K), np.float32)
    x[1, :] = -0.0
    x[2, 5] = 1e-38                       # amax bf16-subnormal-ish: scale is an fp32 subnormal
    x[2, 6] = -3e-39
    x[3, :] = 3.0e38                      # near bf16 max
    x[3, 7] = -1.0
    x[4, :128] = np.float32(17.0 / 128)   # 17 -> tie between 16 and 18 after scaling by amax 3.5
    x[4, 0] = 3.5
    x[5:, :] = np.random.default_rng(0).standard_normal((M - 5, K)).astype(np.float32)
    x[200:210, 128:256] = 0.0             # zero token group
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    fin = bits[np.isfinite(bits)]
    x[128:256, 256:384].flat[: min(fin.size, 128 * 128)] = fin[: 128 * 128]
    xb = workloads.to_bf16(x)
    check_act(xb, scale_mode)
    check_w(xb, scale_mode)


def test_non_finite_inputs():
    """Infinities and NaNs (amax/448 mode).  A group holding an infinity has
    s = inf: its finite values code as signed zeros (x / inf) and its
    infinities as NaN (inf / inf); a NaN codes as NaN (0x7F) in any group,
    and the amax ignores it.  The codes and scales match the oracle's."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((256, 384)).astype(np.float32)
    x[0, 0] = np.inf
    x[0, 1], x[0, 2] = -2.0, -0.0
    x[1, 5], x[1, 6] = np.nan, -np.nan
    x[2, 3] = -np.inf
    x[3, :128] = 0.0
    x[3, 9] = np.nan                      # a group of zeros and one NaN: s = 1
    x[130, 200] = np.inf                  # a token group (rows 128..255) with an infinity
    x[140:150, 300] = np.nan
    xb = workloads.to_bf16(x)
    check_act(xb)
    check_w(xb)


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
def test_every_bf16_bit_pattern(scale_mode):
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    fin = bits[np.isfinite(bits)]
    x = np.zeros((512, 256), np.float32)
    x.flat[: fin.size] = fin
    xb = workloads.to_bf16(x)
    check_act(xb, scale_mode)
    check_w(xb, scale_mode)


@pytest.mark.parametrize("amax", [3.0, 0.7109375, 123.5, 1.0e-30, 5.0e-39, 2.5e38, 3.5, 1.0])
def test_every_bf16_value_below_a_fixed_amax(amax):
    """Each 128-group holds +-amax and then every finite bf16 value of smaller
    magnitude, so x / s sweeps the whole E4M3 range, including values close to
    its rounding boundaries (non-power-of-two scales), fp32-subnormal scales
    (amax 5e-39) and power-of-two scales (amax 3.5, 1.0)."""
    a = np.float32(workloads.to_bf16(np.array([amax], np.float32)).float().numpy()[0])
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = bits[np.isfinite(bits) & (np.abs(bits) <= a)]
    per = 127
    groups = -(-vals.size // per)
    groups += (-groups) % 2                      # an even number of groups -> K = 256 per row
    padded = np.zeros(groups * per, np.float32)
    padded[: vals.size] = vals
    g = padded.reshape(groups, per)
    first = np.where(np.arange(groups) % 2 == 0, a, -a).astype(np.float32)[:, None]
    x = np.concatenate([first, g], axis=1).reshape(-1, 256)
    rows = -(-x.shape[0] // 128) * 128
    full = np.zeros((rows, 256), np.float32)
    full[: x.shape[0]] = x
    xb = workloads.to_bf16(full)
    check_act(xb)
    check_w(xb)


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
def test_every_bf16_value_as_group_amax(scale_mode):
    """Row group g (128 values along K) has amax = the g-th positive finite
    bf16 value, so every scale amax/448 reachable from bf16 inputs is formed
    once (normal and subnormal quotients alike); the other 127 values of the
    group are that amax times uniform(-1, 1), rounded to bf16."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16
    amax = bits.view(np.float32)
    rng = np.random.default_rng(7)
    groups = np.empty((amax.size, 128), np.float32)
    groups[:, 0] = np.where(rng.random(amax.size) < 0.5, amax, -amax)
    groups[:, 1:] = amax[:, None] * rng.uniform(-1, 1, (amax.size, 127)).astype(np.float32)
    xb = workloads.to_bf16(groups)
    # rounding to bf16 can reach the amax but not exceed it
    assert np.all(np.abs(xb.float().numpy()).max(axis=1) == amax)
    n = -(-amax.size // 256) * 256
    full = np.zeros((n, 128), np.float32)
    full[: amax.size] = xb.float().numpy()
    x = workloads.to_bf16(full.reshape(-1, 256))
    check_act(x, scale_mode)


@pytest.mark.parametrize("name,tag", [("mlp_gateup", "x"), ("mlp_gateup", "w"), ("mlp_down", "x"),
                                      ("mlp_down", "w"), ("mlp_down", "dy"), ("attn_proj", "x"),
                                      ("attn_proj", "w_qkv"), ("attn_proj", "dy_qkv")])
def test_full_size_configs(name, tag):
    t = bf16_input(name, tag)
    if tag.startswith("w"):
        check_w(t)
    else:
        check_act(t)


def test_stack_layer_tensors():
    wl = workloads.make("stack28")
    check_act(workloads.tensor(wl, "x_f"))
    check_act(workloads.tensor(wl, "dy_gu"))
    check_w(workloads.tensor(wl, "w_gu", layer=27))


# ---------------------------------------------------------------- power of two


@pytest.mark.parametrize("amax", [3.0, 3.5, 0.7109375, 1.0e-30, 5.0e-39, 2.5e38, 448.0, 449.0])
def test_pow2_every_bf16_value_below_a_fixed_amax(amax):
    """As the amax/448 sweep, with power-of-two scales: x / s is exact, and
    amax 5e-39 gives a scale below 2^-127, which takes the division path."""
    a = np.float32(workloads.to_bf16(np.array([amax], np.float32)).float().numpy()[0])
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = bits[np.isfinite(bits) & (np.abs(bits) <= a)]
    per = 127
    groups = -(-vals.size // per)
    groups += (-groups) % 2
    padded = np.zeros(groups * per, np.float32)
    padded[: vals.size] = vals
    g = padded.reshape(groups, per)
    first = np.where(np.arange(groups) % 2 == 0, a, -a).astype(np.float32)[:, None]
    x = np.concatenate([first, g], axis=1).reshape(-1, 256)
    rows = -(-x.shape[0] // 128) * 128
    full = np.zeros((rows, 256), np.float32)
    full[: x.shape[0]] = x
    xb = workloads.to_bf16(full)
    check_act(xb, "pow2")
    check_w(xb, "pow2")


@pytest.mark.parametrize("name,tag", [("mlp_gateup", "x"), ("mlp_down", "dy"), ("attn_proj", "w_qkv")])
def test_pow2_full_size_configs(name, tag):
    t = bf16_input(name, tag)
    if tag.startswith("w"):
        check_w(t, "pow2")
    else:
        check_act(t, "pow2")


def test_pow2_linear_layer_against_oracle():
    """Power-of-two scales flow through the unchanged GEMM: FPROP of a
    pow2-quantised layer matches the oracle's GEMM on the oracle's own pow2
    quantisation within the GEMM tolerance."""
    from gpu_helpers import REL_FRO_TOL, rel_fro
    from oracle import gemm as ogemm
    x, w = bf16_input("tiny", "x"), bf16_input("tiny", "w")
    Xq, sX, _, _ = ops.quantize_act_1x128(x.to(dev()), rows=True, tokens=False, scale_mode="pow2")
    Wq, _, sW = ops.quantize_w_128x128(w.to(dev()), want_qT=False, scale_mode="pow2")
    Y = ops.fp8_block_gemm(ops.FPROP, Xq, sX, Wq, sW)
    assert ops.sync_status() == 0
    oq, os_ = quant.quantize_act_1x128(np32(x), scale_mode="pow2")
    wq, _, ws = quant.quantize_w_128x128(np32(w), scale_mode="pow2")
    want = ogemm.fprop(oq, os_, wq, ws)[1]
    assert rel_fro(np32(Y), want) <= REL_FRO_TOL


# ------------------------------------------------------- reciprocal multiply


def _below_amax_groups(amax):
    """Groups of 256 columns: +-amax, then every finite bf16 value of smaller
    magnitude (127 per 128-group), zero-padded to whole tiles."""
    a = np.float32(workloads.to_bf16(np.array([amax], np.float32)).float().numpy()[0])
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = bits[np.isfinite(bits) & (np.abs(bits) <= a)]
    per = 127
    groups = -(-vals.size // per)
    groups += (-groups) % 2
    padded = np.zeros(groups * per, np.float32)
    padded[: vals.size] = vals
    g = padded.reshape(groups, per)
    first = np.where(np.arange(groups) % 2 == 0, a, -a).astype(np.float32)[:, None]
    x = np.concatenate([first, g], axis=1).reshape(-1, 256)
    rows = -(-x.shape[0] // 128) * 128
    full = np.zeros((rows, 256), np.float32)
    full[: x.shape[0]] = x
    return workloads.to_bf16(full)


@pytest.mark.parametrize("amax", [13.0, 3.0, 0.7109375, 123.5, 1.0e-30, 5.0e-39, 2.5e38, 1.0])
def test_mul_recip_every_bf16_value_below_a_fixed_amax(amax):
    """The sweep of the amax/448 mode with codes from x * fp32(448/amax): the
    products land on and around E4M3 midpoints (amax 13 puts x = 39 * 2^-16
    exactly on one before rounding), and amax 5e-39 saturates the
    multiplier at the largest finite fp32."""
    xb = _below_amax_groups(amax)
    check_act(xb, "mul_recip")
    check_w(xb, "mul_recip")


@pytest.mark.parametrize("name,tag", [("mlp_gateup", "x"), ("mlp_down", "dy"), ("attn_proj", "w_qkv")])
def test_mul_recip_full_size_configs(name, tag):
    t = bf16_input(name, tag)
    if tag.startswith("w"):
        check_w(t, "mul_recip")
    else:
        check_act(t, "mul_recip")


def test_mul_recip_linear_layer_against_oracle():
    """The reciprocal-multiply mode through the fused linear entry points:
    saved FP8 tensors and scales bit-exact against the oracle's composed
    linear in the same mode, outputs within the GEMM tolerance."""
    from gpu_helpers import REL_FRO_TOL, rel_fro
    from oracle import gemm as ogemm
    rng = np.random.default_rng(41)
    X = workloads.to_bf16(rng.standard_normal((384, 640)).astype(np.float32))
    W = workloads.to_bf16((rng.standard_normal((512, 640)) * 0.02).astype(np.float32))
    dY = workloads.to_bf16((rng.standard_normal((384, 512)) * 1e-3).astype(np.float32))
    Y, saved = ops.linear_fwd(X.to(dev()), W.to(dev()), scale_mode="mul_recip")
    dX, dW = ops.linear_bwd(dY.to(dev()), saved, scale_mode="mul_recip")
    assert ops.sync_status() == 0
    oY, osaved = ogemm.linear_fwd(np32(X), np32(W), scale_mode="mul_recip")
    for k in ("WqT", "XqT"):
        assert_codes_equal(u8(saved[k]), osaved[k], k)
    for k in ("sW", "sXT"):
        assert_scales_equal(saved[k].cpu().numpy(), osaved[k], k)
    assert rel_fro(np32(Y), oY) <= REL_FRO_TOL
    odX, odW = ogemm.linear_bwd(np32(dY), osaved, scale_mode="mul_recip")
    assert rel_fro(np32(dX), odX) <= REL_FRO_TOL
    assert rel_fro(np32(dW), odW) <= REL_FRO_TOL
    # the same layer in the default mode differs only in a few codes
    _, saved_d = ops.linear_fwd(X.to(dev()), W.to(dev()))
    assert torch.equal(saved_d["sXT"], saved["sXT"]) and torch.equal(saved_d["sW"], saved["sW"])
    step = (u8(saved_d["XqT"]) & 0x7F).astype(int) - (u8(saved["XqT"]) & 0x7F).astype(int)
    assert np.abs(step).max() <= 1


def test_unknown_scale_mode_is_rejected():
    from blockwise_fp8_linear_quantise_b300 import _lib
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device=dev())
    q = torch.empty((128, 128), dtype=torch.uint8, device=dev())
    s = torch.empty((1, 128), dtype=torch.float32, device=dev())
    st = torch.cuda.current_stream().cuda_stream
    for bad in (3, 7, -1):
        assert _lib.load().bfp8_quantize_act_1x128_ex(x.data_ptr(), 128, 128, q.data_ptr(), s.data_ptr(), None,
                                                      None, bad, st) == 1


def test_weight_block_worked_example_on_gpu():
    """The hand-worked 256 x 256 weight fixture: block scales and the listed
    codes, in both the fprop (Wq) and dgrad (WqT) layouts."""
    from test_oracle_quant import golden_weight_block
    w, scales, codes = golden_weight_block()
    q, qT, s = ops.quantize_w_128x128(to_gpu(w, torch.bfloat16))
    assert ops.sync_status() == 0
    s = s.cpu().numpy()
    for (bi, bj), bits in scales.items():
        assert s[bi, bj].view(np.uint32) == bits, (bi, bj)
    qn, qTn = u8(q), u8(qT)
    for (ii, jj), (_, code) in codes.items():
        assert qn[ii, jj] == code and qTn[jj, ii] == code, (ii, jj)
    check_w(torch.from_numpy(w).to(torch.bfloat16))


def test_stack_weights_all_layers():
    """Every weight of the 28-layer stack (QKV, O, gate+up, down per layer),
    as the benchmark's step quantises them, bit-exact against the oracle (run
    over the host's cores; it changes no bit)."""
    from oracle import parallel
    wl = workloads.make("stack28")
    try:
        for layer in range(28):
            for tag in ("w_qkv", "w_o", "w_gu", "w_down"):
                w = workloads.tensor(wl, tag, layer)
                q, qT, s = ops.quantize_w_128x128(w.to(dev()))
                assert ops.sync_status() == 0
                oq, oqT, os_ = parallel.quantize_w_128x128(np32(w))
                assert_codes_equal(u8(q), oq, f"Wq {tag} layer {layer}")
                assert_codes_equal(u8(qT), oqT, f"WqT {tag} layer {layer}")
                assert_scales_equal(s.cpu().numpy(), os_, f"sW {tag} layer {layer}")
    finally:
        parallel.shutdown()


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
@pytest.mark.parametrize("outputs", ["both", "q", "qT"])
def test_weight_batch_matches_the_oracle(scale_mode, outputs):
    """Six weights of different shapes (two launches: four, then two) quantised
    by bfp8_quantize_w_128x128_batch: every job's codes and scales equal the
    oracle's and those of its own single call, bit for bit."""
    shapes = [(512, 256), (256, 256), (1536, 256), (256, 768), (128, 128), (384, 640)]
    rng = np.random.default_rng(31)
    ws = [workloads.to_bf16((rng.standard_normal(sh) * np.exp2(rng.integers(-8, 8))).astype(np.float32))
          for sh in shapes]
    want_q, want_qT = outputs in ("both", "q"), outputs in ("both", "qT")
    got = ops.quantize_w_batch([w.to(dev()) for w in ws], want_q=want_q, want_qT=want_qT, scale_mode=scale_mode)
    assert ops.sync_status() == 0
    for w, (q, qT, s) in zip(ws, got):
        oq, oqT, os_ = quant.quantize_w_128x128(np32(w), scale_mode=scale_mode)
        assert_scales_equal(s.cpu().numpy(), os_, "sW")
        if want_q:
            assert_codes_equal(u8(q), oq, "Wq")
        if want_qT:
            assert_codes_equal(u8(qT), oqT, "WqT")
        sq, sqT, ss = ops.quantize_w_128x128(w.to(dev()), want_q=want_q, want_qT=want_qT, scale_mode=scale_mode)
        assert torch.equal(ss, s) and (not want_q or torch.equal(sq, q)) and (not want_qT or torch.equal(sqT, qT))


def test_weight_batch_on_one_stack_layer():
    """The four weights of one stack28 layer (QKV, O, gate+up, down), as the
    step quantises them: one launch, bit-exact against the oracle."""
    wl = workloads.make("stack28")
    tags = []
    for s in wl.linears:
        if workloads.layer_of(s) == 3 and s.w_tag not in tags:
            tags.append(s.w_tag)
    ws = [workloads.tensor(wl, t, 3) for t in tags]
    assert len(ws) == 4
    got = ops.quantize_w_batch([w.to(dev()) for w in ws])
    assert ops.sync_status() == 0
    for w, (q, qT, s) in zip(ws, got):
        oq, oqT, os_ = quant.quantize_w_128x128(np32(w))
        assert_codes_equal(u8(q), oq, "Wq")
        assert_codes_equal(u8(qT), oqT, "WqT")
        assert_scales_equal(s.cpu().numpy(), os_, "sW")
