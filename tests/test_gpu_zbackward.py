"""The backward data gradient dX = dY W of the FP8 linear layer (E4M3 in the
backward pass as well: the Float8 paragraph of the 88811315.cn post), built
from the library's forward calls: dY quantised by fp8bs_act_quant (1x128
groups along N, the contraction dimension), the weight's transpose
quantised by fp8bs_weight_quant (its 128x128 blocks are W's blocks
transposed, with the same amax, so its codes are W's codes transposed), and
fp8bs_gemm.  Checked against the oracle's dgrad within the GEMM bound."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_gemm_close, dev_bf16, host, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


@pytest.mark.parametrize("M,N,K", [(300, 512, 768), (4096, 576 + 64, 7168)])
def test_dgrad_through_the_forward_gemm(F, orc, M, N, K):
    """Reduced shape, then the KV down-projection's backward (W [640 (576
    padded to whole blocks), 7168], 4096 tokens) on sampled rows."""
    rng = np.random.default_rng(M + N)
    dy = synth.activations(rng, M, N, n_outlier=4, outlier_scale=10.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    dyq, sdy = F.fp8bs_act_quant(dev_bf16(dy))
    wtq, swt = F.fp8bs_weight_quant(dev_bf16(np.ascontiguousarray(w.T)))   # [K, N], grid [K/128, N/128]
    dx = F.fp8bs_gemm(dyq, sdy, wtq, swt)                                 # [M, K]
    assert F.fp8bs_sync_status() == 0
    wq_o, sw_o = orc.weight_quant(w)
    assert np.array_equal(host(wtq), np.ascontiguousarray(wq_o.T))
    assert np.array_equal(host(swt).view(np.uint32), np.ascontiguousarray(sw_o.T).view(np.uint32))
    rows = np.arange(M) if M <= 512 else sample_rows(M, 24, seed=5)
    dyq_o, sdy_o = orc.act_quant(dy[rows])
    dx_ref, L = orc.gemm_dgrad(dyq_o, sdy_o, wq_o, sw_o)
    assert_gemm_close(host(dx)[rows], dx_ref, L, f"dgrad {M}x{N}x{K}")
