"""The backward weight gradient dW = dY^T X of the FP8 linear layer (E4M3 in
the backward pass as well: the Float8 paragraph of the 88811315.cn post),
on the device: fp8bs_act_quant_cols (128x1 groups along the tokens, codes
written transposed) bit for bit against the oracle's column quantisation,
and fp8bs_gemm_wgrad against the oracle's wgrad within the GEMM bound
|dw - dw_ref| <= 2^-8 |dw_ref| + 1e-4 sum_m |a_m b_m| (fp32 output)."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_bits_equal, dev_bf16, host
from oracle import gemm_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _cols(F, orc, x):
    M, K = x.shape
    xqt, sc = F.fp8bs_act_quant_cols(dev_bf16(x))
    assert F.fp8bs_sync_status() == 0
    xq_o, sc_o = orc.act_quant_cols(x)
    assert_bits_equal(host(xqt)[:, :M], np.ascontiguousarray(xq_o.T), f"codes {M}x{K}")
    assert_bits_equal(host(sc), sc_o, f"scales {M}x{K}")
    return xqt, sc, xq_o, sc_o


@pytest.mark.parametrize("M,K", [(1, 64), (128, 64), (300, 256), (257, 1536), (4096, 576), (1000, 7168)])
def test_act_quant_cols_bit_exact(F, orc, M, K):
    rng = np.random.default_rng(M + K)
    x = synth.activations(rng, M, K, n_outlier=min(4, K // 64), outlier_scale=30.0)
    _cols(F, orc, x)


def test_act_quant_cols_special_blocks(F, orc):
    """All-zero columns (s = 0, +-0 codes with the input's sign), a column of
    one nonzero value, a ragged last block whose amax sits in its last row."""
    M, K = 200, 128
    rng = np.random.default_rng(3)
    x = synth.activations(rng, M, K).astype(np.uint16)
    x[:, 0] = 0x0000
    x[:, 1] = 0x8000          # -0.0
    x[:, 2] = 0
    x[5, 2] = synth.to_bf16_bits(np.array([3.0], dtype=np.float32))[0]
    x[199, 3] = synth.to_bf16_bits(np.array([1000.0], dtype=np.float32))[0]
    _cols(F, orc, x)


@pytest.mark.parametrize("M,K", [(333, 192), (16, 64)])
def test_act_quant_cols_strided_padding_untouched(F, orc, M, K):
    """x, xqt and sc as views with row strides wider than their rows: the
    codes and scales land at their strides, and nothing past M tokens in a
    code row (the ragged last block's tail) or past K in a scale row is
    written."""
    rng = np.random.default_rng(M * 7 + K)
    x = synth.activations(rng, M, K, n_outlier=min(3, K // 64), outlier_scale=30.0)
    xb = torch.zeros((M, K + 128), dtype=torch.bfloat16, device="cuda")
    xb[:, :K] = dev_bf16(x)
    ldt = (M + 15) // 16 * 16 + 48
    xqt_buf = torch.full((K, ldt), 0x5A, dtype=torch.uint8, device="cuda")
    sc_buf = torch.full(((M + 127) // 128, K + 8), -7.0, dtype=torch.float32, device="cuda")
    xqt, sc = F.fp8bs_act_quant_cols(xb[:, :K], xqt=xqt_buf, sc=sc_buf[:, :K])
    assert F.fp8bs_sync_status() == 0
    xq_o, sc_o = orc.act_quant_cols(x)
    got = host(xqt_buf)
    assert_bits_equal(got[:, :M], np.ascontiguousarray(xq_o.T), f"codes {M}x{K}")
    assert (got[:, M:] == 0x5A).all(), "code bytes past M written"
    sc_h = host(sc_buf)
    assert_bits_equal(np.ascontiguousarray(sc_h[:, :K]), sc_o, f"scales {M}x{K}")
    assert (sc_h[:, K:] == -7.0).all(), "scales past K written"


def _wgrad(F, orc, orc_mt, T, N, K, seed, rows=None):
    rng = np.random.default_rng(seed)
    dy = synth.activations(rng, T, N, n_outlier=4, outlier_scale=10.0)
    x = synth.activations(rng, T, K, n_outlier=4, outlier_scale=20.0)
    dyqt, sdy, dyq_o, sdy_o = _cols(F, orc, dy)
    xqt, sx, xq_o, sx_o = _cols(F, orc, x)
    dw = F.fp8bs_gemm_wgrad(dyqt, sdy, xqt, sx, T)
    assert F.fp8bs_sync_status() == 0
    dw_h = host(dw)
    dw_ref, L = orc_mt.gemm_wgrad(dyq_o, sdy_o, xq_o, sx_o, rows=rows)
    got = dw_h if rows is None else dw_h[rows]
    err = np.abs(got.astype(np.float64) - dw_ref)
    tol = gemm_tolerance(dw_ref, L)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"wgrad {T}x{N}x{K}: {len(bad)} outside the bound, first {bad[:3].tolist()}"
    return dw


@pytest.mark.parametrize("T,N,K", [(128, 128, 192), (300, 256, 384), (1000, 192, 512), (129, 320, 1024)])
def test_wgrad_small_every_element(F, orc, orc_mt, T, N, K):
    _wgrad(F, orc, orc_mt, T, N, K, seed=T + N + K)


def test_wgrad_kv_down_backward(F, orc, orc_mt):
    """The KV down-projection's weight gradient: dY [4096, 576], X [4096, 7168]
    (W [576, 7168]); every row of dW, every column."""
    _wgrad(F, orc, orc_mt, 4096, 576, 7168, seed=11)


def test_wgrad_deterministic(F, orc, orc_mt):
    a = _wgrad(F, orc, orc_mt, 300, 256, 384, seed=5)
    b = _wgrad(F, orc, orc_mt, 300, 256, 384, seed=5)
    assert torch.equal(a, b)
