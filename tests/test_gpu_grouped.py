"""GPU parity of fp8bs_grouped_gemm (variable-M per-expert batches)."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_gemm_close, dev, dev_bf16, host, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _grouped_small(F, orc, counts, N, K, seed):
    rng = np.random.default_rng(seed)
    counts = np.asarray(counts)
    G = counts.size
    off = synth.offsets_from_counts(counts)
    T = int(off[-1])
    x = synth.activations(rng, max(T, 1), K, n_outlier=4, outlier_scale=20.0)[:T]
    w = synth.normal_bf16(rng, (G, N, K), 0.02)
    xq, sx = orc.act_quant(x, lds=max(4, (K // 128 + 3) // 4 * 4))
    wqs, sws = zip(*[orc.weight_quant(w[g]) for g in range(G)])
    wq, sw = np.stack(wqs), np.stack(sws)
    ld = (N + 7) // 8 * 8  # the C ABI wants a row stride that is a multiple of 8
    y = torch.full((T, ld), 7.0, dtype=torch.bfloat16, device="cuda")[:, :N]
    F.fp8bs_grouped_gemm(dev(xq), dev(sx), dev(wq), dev(sw), dev(off), y=y)
    assert F.fp8bs_sync_status() == 0
    y_ref, L = orc.grouped_gemm(xq, sx, wq, sw, off)
    yh = host(y.contiguous())
    assert_gemm_close(yh, y_ref, L, f"grouped {counts.tolist()}")


@pytest.mark.parametrize("counts,N,K", [
    ([3, 0, 130, 1, 0, 257], 256, 256),
    ([128, 128], 128, 128),
    ([0, 0, 5], 576, 384),
    ([1000], 136, 256),
    ([0] * 7 + [40] + [0] * 8, 130, 128),
])
def test_grouped_small(F, orc, counts, N, K):
    _grouped_small(F, orc, counts, N, K, seed=len(counts) + N)


def test_grouped_token_tile_edges(F, orc):
    """Experts whose row counts sit on the edges of the token tiles (16-row
    MMA width steps, 32-row load boxes, the two 128-column promotion halves,
    256-row tiles)."""
    counts = [1, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 511, 0, 2]
    _grouped_small(F, orc, counts, 256, 256, seed=17)


def test_grouped_many_experts(F, orc):
    rng = np.random.default_rng(3)
    counts = rng.poisson(60, size=64)
    counts[::9] = 0
    _grouped_small(F, orc, counts, 256, 512, seed=4)


def test_grouped_matches_dense_per_expert(F, orc):
    """Grouped output rows == dense fp8bs_gemm on each expert's slice."""
    rng = np.random.default_rng(5)
    counts = np.array([70, 0, 200, 129])
    off = synth.offsets_from_counts(counts)
    K, N = 384, 256
    x = synth.activations(rng, int(off[-1]), K)
    w = synth.normal_bf16(rng, (4, N, K), 0.02)
    xq, sx = F.fp8bs_act_quant(dev_bf16(x))
    wq = torch.empty((4, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((4, 2, 3), dtype=torch.float32, device="cuda")
    for g in range(4):
        F.fp8bs_weight_quant(dev_bf16(w[g]), wq=wq[g], sw=sw[g])
    y = F.fp8bs_grouped_gemm(xq, sx, wq, sw, dev(off))
    for g in range(4):
        r0, r1 = int(off[g]), int(off[g + 1])
        if r1 > r0:
            yd = F.fp8bs_gemm(xq[r0:r1].contiguous(), sx[r0:r1].contiguous(), wq[g], sw[g])
            assert F.fp8bs_sync_status() == 0
            # same chunk sums and promotion order: bit-identical
            assert torch.equal(y[r0:r1].view(torch.int16), yd.view(torch.int16))


def test_moe_full_config_every_row(F, orc, orc_mt):
    """The MoE configuration at full size (4096 tokens, 256 experts, top-8,
    N=2048, K=7168): device pipeline vs the oracle's pipeline on every row of
    every expert (each expert's weight quantised by the oracle from the same
    bf16 bits, its GEMM in the oracle's OpenMP build)."""
    case = synth.moe()
    T = int(case.offsets[-1])
    assert T == 4096 * 8
    G, N, K = case.n_experts, case.n, case.k
    x_rows = case.x_rows
    xq, sx = F.fp8bs_act_quant(dev_bf16(x_rows))
    wq = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
    for g in range(G):
        F.fp8bs_weight_quant(synth.expert_weight(case, g, "cuda"), wq=wq[g], sw=sw[g])
    off_d = dev(case.offsets)
    y = F.fp8bs_grouped_gemm(xq, sx, wq, sw, off_d)
    assert F.fp8bs_sync_status() == 0
    yh = host(y)
    del xq, sx, wq, sw, y
    xq_o, sx_o = orc.act_quant(x_rows)
    checked = 0
    for g in range(G):
        r0, r1 = int(case.offsets[g]), int(case.offsets[g + 1])
        if r1 == r0:
            continue
        wb = synth.expert_weight(case, g, "cuda").view(torch.int16).cpu().numpy().view(np.uint16)
        wq_o, sw_o = orc.weight_quant(wb)
        y_ref, L = orc_mt.gemm(xq_o[r0:r1], sx_o[r0:r1], wq_o, sw_o)
        assert_gemm_close(yh[r0:r1], y_ref, L, f"moe expert {g}")
        checked += r1 - r0
    assert checked == T
