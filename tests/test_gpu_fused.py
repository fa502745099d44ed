"""GPU parity of fp8bs_gemm_fused: the bias add of linear() and the output
re-quantised to FP8 ("DeepSeek-V3" repository overview, "FP8 混合精度训练").

y is checked against the oracle's fp64 GEMM plus bias with the GEMM bound.
The FP8 output is checked two ways: bit-identical to fp8bs_act_quant applied
to the same call's bf16 y (the same quantisation, whose exactness against the
oracle the quantiser tests establish), and, dequantised, against the oracle's
y within the GEMM bound plus the e4m3 rounding bound.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_gemm_close, dev, dev_bf16, host
from oracle import gemm_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _operands(orc, M, N, K, seed):
    rng = np.random.default_rng(seed)
    x = synth.activations(rng, M, K, n_outlier=min(8, K // 64), outlier_scale=20.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    bias = synth.normal_bf16(rng, (N,), 0.5)
    xq, sx = orc.act_quant(x, lds=max(4, (K // 128 + 3) // 4 * 4))
    wq, sw = orc.weight_quant(w)
    return xq, sx, wq, sw, bias


def _check_fp8_out(yq, sy, y_ref, L, what):
    """dec(yq) * sy against the oracle's y: the GEMM bound on y, then at most
    half an e4m3 step (2^-4 relative for normal codes, 2^-10 * s below)."""
    v = synth_e4m3_values()
    N = y_ref.shape[1]
    s = np.repeat(sy.astype(np.float64), 128, axis=1)[:, :N]
    deq = v[yq] * s
    tol = gemm_tolerance(y_ref, L)
    # (+ 2^-20 relative for the fp32 rounding of the quotient before encoding)
    bound = tol + np.ldexp(np.abs(y_ref) + tol, -4) * (1 + 2.0 ** -20) + np.ldexp(s, -10) + 1e-30
    bad = np.abs(deq - y_ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} fp8 outputs outside the bound"


def synth_e4m3_values():
    import ml_dtypes
    return np.arange(256, dtype=np.uint8).view(ml_dtypes.float8_e4m3fn).astype(np.float64)


# 148 SMs: the cost model picks 256, 192 and 160 columns for these (see
# test_gpu_gemm.test_gemm_tile_widths); with fp8 output the call always
# takes 256-column tiles.
WIDTH_SHAPES = [(4000, 1000, 384), (4000, 700, 384), (4000, 1200, 256)]


@pytest.mark.parametrize("M,N,K", WIDTH_SHAPES + [(5, 130, 256), (300, 576, 640)])
def test_fused_bias(F, orc, orc_mt, M, N, K):
    xq, sx, wq, sw, bias = _operands(orc, M, N, K, seed=M + N)
    y, yq, sy = F.fp8bs_gemm_fused(dev(xq), dev(sx), dev(wq), dev(sw), bias=dev_bf16(bias))
    assert yq is None and sy is None
    assert F.fp8bs_sync_status() == 0
    y_ref, L = orc_mt.gemm(xq, sx, wq, sw, bias=bias)
    assert_gemm_close(host(y), y_ref, L, f"fused bias {M}x{N}x{K}")


def test_fused_without_bias_equals_gemm(F, orc):
    """No bias, bf16 out only: the same kernel and plan as fp8bs_gemm without a
    workspace, so the outputs are identical bit for bit."""
    M, N, K = 4000, 1200, 256
    xq, sx, wq, sw, _ = _operands(orc, M, N, K, seed=3)
    a = dev(xq), dev(sx), dev(wq), dev(sw)
    y_fused, _, _ = F.fp8bs_gemm_fused(*a)
    y_plain = F.fp8bs_gemm(*a)
    assert F.fp8bs_sync_status() == 0
    assert np.array_equal(host(y_fused), host(y_plain))


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (129, 256, 384), (700, 1536, 1024), (4000, 1024, 256)])
def test_fused_fp8_out(F, orc, orc_mt, M, N, K):
    xq, sx, wq, sw, bias = _operands(orc, M, N, K, seed=2 * M + N)
    a = dev(xq), dev(sx), dev(wq), dev(sw)
    y, yq, sy = F.fp8bs_gemm_fused(*a, bias=dev_bf16(bias), want_fp8=True)
    _, yq_only, sy_only = F.fp8bs_gemm_fused(*a, bias=dev_bf16(bias), want_y=False, want_fp8=True)
    xq2, sx2 = F.fp8bs_act_quant(y)
    assert F.fp8bs_sync_status() == 0
    yq_h, sy_h = host(yq), host(sy)
    # the same quantisation as act_quant on this call's y, bit for bit
    assert np.array_equal(yq_h, host(xq2))
    assert np.array_equal(sy_h.view(np.uint32), host(sx2)[:, : N // 128].view(np.uint32))
    # without y the fp8 output is the same
    assert np.array_equal(host(yq_only), yq_h)
    assert np.array_equal(host(sy_only).view(np.uint32), sy_h.view(np.uint32))
    # against the oracle, every element
    y_ref, L = orc_mt.gemm(xq, sx, wq, sw, bias=bias)
    assert_gemm_close(host(y), y_ref, L, f"fused y {M}x{N}x{K}")
    _check_fp8_out(yq_h, sy_h, y_ref, L, f"fused fp8 {M}x{N}x{K}")


def test_fused_q_down_full(F, orc, orc_mt):
    """The q down-projection at M = 4096 (N = 1536 = 12 output groups):
    device pipeline (weight_quant, act_quant, fused GEMM with bias and fp8
    output) against the oracle's pipeline on every element."""
    case = synth.q_down(4096)
    M, N, K = case.shape
    rng = np.random.default_rng(31)
    bias = synth.normal_bf16(rng, (N,), 0.5)
    wq, sw = F.fp8bs_weight_quant(dev_bf16(case.w))
    xq, sx = F.fp8bs_act_quant(dev_bf16(case.x))
    y, yq, sy = F.fp8bs_gemm_fused(xq, sx, wq, sw, bias=dev_bf16(bias), want_fp8=True)
    assert F.fp8bs_sync_status() == 0
    xq_o, sx_o = orc.act_quant(case.x)
    wq_o, sw_o = orc.weight_quant(case.w)
    y_ref, L = orc_mt.gemm(xq_o, sx_o, wq_o, sw_o, bias=bias)
    assert_gemm_close(host(y), y_ref, L, "q_down fused y")
    _check_fp8_out(host(yq), host(sy), y_ref, L, "q_down fused fp8")
