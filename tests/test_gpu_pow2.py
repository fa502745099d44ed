"""Power-of-two (UE8M0-style) scales on the device -- the scale_fmt reading of
the pages' act_quant ("DeepSeek-V3" repository overview, the linear()
excerpt): fp8bs_act_quant_pow2 and fp8bs_weight_quant_pow2 bit for bit
against the oracle's power-of-two quantisers, and the power-of-two operands
through fp8bs_gemm against the oracle's GEMM within the GEMM bound."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_bits_equal, assert_gemm_close, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _act(F, orc, x):
    xq, sx = F.fp8bs_act_quant_pow2(dev_bf16(x))
    assert F.fp8bs_sync_status() == 0
    xq_o, sx_o = orc.act_quant_pow2(x)
    K = x.shape[1]
    assert_bits_equal(host(xq), xq_o, "pow2 codes")
    assert_bits_equal(host(sx)[:, :K // 128], sx_o[:, :K // 128], "pow2 scales")


@pytest.mark.parametrize("M,K", [(1, 128), (5, 512), (300, 1024), (4096, 7168)])
def test_act_quant_pow2_bit_exact(F, orc, M, K):
    rng = np.random.default_rng(M + K)
    _act(F, orc, synth.activations(rng, M, K, n_outlier=min(8, K // 64), outlier_scale=30.0))


def test_act_quant_pow2_every_bf16_amax(F, orc):
    """One group per positive finite bf16 value a (subnormals included): a
    itself and 127 values below it, so every exponent and the 1.75 mantissa
    boundary of the scale rule are taken, with tiny groups on the
    IEEE-division path."""
    amax = np.arange(1, 0x7F80, dtype=np.uint16)           # +subnormals .. largest finite
    rng = np.random.default_rng(7)
    a = synth.bf16_bits_to_f32(amax).astype(np.float32)
    frac = rng.random((amax.size, 127), dtype=np.float32)
    rest = synth.to_bf16_bits((a[:, None] * frac).astype(np.float32))
    rest = np.where(synth.bf16_bits_to_f32(rest) <= a[:, None], rest, amax[:, None])  # keep |x| <= a
    sign = (rng.random((amax.size, 127)) < 0.5).astype(np.uint16) << 15
    x = np.concatenate([amax[:, None], rest | sign], axis=1)
    _act(F, orc, x)


@pytest.mark.parametrize("N,K", [(128, 128), (200, 384), (576, 7168), (7168, 7168)])
def test_weight_quant_pow2_bit_exact(F, orc, N, K):
    rng = np.random.default_rng(N + K)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    w[0, 0] = synth.to_bf16_bits(np.array([3.5], dtype=np.float32))[0]   # one outlier block
    wq, sw = F.fp8bs_weight_quant_pow2(dev_bf16(w))
    assert F.fp8bs_sync_status() == 0
    wq_o, sw_o = orc.weight_quant_pow2(w)
    assert_bits_equal(host(wq), wq_o, "pow2 weight codes")
    assert_bits_equal(host(sw), sw_o, "pow2 weight scales")


def test_gemm_on_pow2_operands(F, orc, orc_mt):
    """Power-of-two scales are ordinary fp32 scales to fp8bs_gemm: the
    device pipeline (pow2 quantisers, then the GEMM) against the oracle's."""
    rng = np.random.default_rng(21)
    M, N, K = 1000, 1536, 7168
    x = synth.activations(rng, M, K, n_outlier=8, outlier_scale=25.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    xq, sx = F.fp8bs_act_quant_pow2(dev_bf16(x))
    wq, sw = F.fp8bs_weight_quant_pow2(dev_bf16(w))
    y = F.fp8bs_gemm(xq, sx, wq, sw)
    assert F.fp8bs_sync_status() == 0
    xq_o, sx_o = orc.act_quant_pow2(x)
    wq_o, sw_o = orc.weight_quant_pow2(w)
    y_ref, L = orc_mt.gemm(xq_o, sx_o, wq_o, sw_o)
    assert_gemm_close(host(y), y_ref, L, "gemm on pow2 operands")
