"""GPU parity of fp8bs_gemm against the oracle's exact fp64 block GEMM.

Small cases: the GEMM alone, fed the oracle's quantised operands, compared on
every element.  Full-size cases (the bench's shapes and launch): the whole
pipeline (weight_quant, act_quant, gemm) on the device from the synthetic bf16
inputs, against the oracle's pipeline on the same inputs, on every element
(the oracle's GEMM in its OpenMP build, row chunks at a time).
Bound: |y - y_ref| <= 2^-8 |y_ref| + 1e-4 sum_k |a_k b_k|.
"""
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


def _gemm_only(F, orc, xbits, wbits, workspace=True, rows=None):
    xq, sx = orc.act_quant(xbits, lds=max(4, (xbits.shape[1] // 128 + 3) // 4 * 4))
    wq, sw = orc.weight_quant(wbits)
    M, N, K = xq.shape[0], wq.shape[0], xq.shape[1]
    ws = None
    if workspace:
        n = F.fp8bs_gemm_workspace_size(M, N, K)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None
    y = F.fp8bs_gemm(dev(xq), dev(sx), dev(wq), dev(sw), workspace=ws)
    assert F.fp8bs_sync_status() == 0
    y_ref, L = orc.gemm(xq, sx, wq, sw, rows=rows)
    yh = host(y) if rows is None else host(y)[rows]
    return assert_gemm_close(yh, y_ref, L, f"gemm {M}x{N}x{K}"), host(y)


def test_gemm_tiny(F, orc):
    c = synth.tiny()
    _gemm_only(F, orc, c.x, c.w)


@pytest.mark.parametrize("M,N,K", [
    (1, 128, 128), (1, 576, 512), (5, 130, 256), (128, 128, 128), (129, 256, 384),
    (300, 576, 640), (64, 1536, 1024), (256, 8, 256), (200, 1000, 1152), (1000, 136, 128),
])
def test_gemm_ragged_shapes(F, orc, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    x = synth.activations(rng, M, K, n_outlier=min(8, K // 64), outlier_scale=25.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    _gemm_only(F, orc, x, w)


@pytest.mark.parametrize("M,N,K", [
    # 148 SMs, relative chunk periods 256 -> 1.00, 192 -> 0.91, 160 -> 0.77:
    # 256 columns 32 x 4 = 128 tiles (one wave) against 192: 32 x 6 = 192 and
    # 160: 32 x 7 = 224 (two waves each) -> the 256-column kernel
    (4000, 1000, 384),
    # 256: 32 x 3 = 96 and 192: 32 x 4 = 128 tiles (one wave), 160: 160 tiles
    # (two) -> the 192-column kernel (three promotion warpgroups)
    (4000, 700, 384),
    # 256: 160, 192: 224, 160: 256 tiles, two waves each -> the 160-column
    # kernel, persistent CTAs taking two tiles
    (4000, 1200, 256),
])
def test_gemm_tile_widths(F, orc, orc_mt, M, N, K):
    """Shapes picked so that each tile width runs over several CTAs (each
    taking several tiles) with ragged edges; every element is compared."""
    rng = np.random.default_rng(M + N + K)
    x = synth.activations(rng, M, K, n_outlier=4, outlier_scale=25.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    xq, sx = orc.act_quant(x, lds=max(4, (K // 128 + 3) // 4 * 4))
    wq, sw = orc.weight_quant(w)
    y = F.fp8bs_gemm(dev(xq), dev(sx), dev(wq), dev(sw))
    assert F.fp8bs_sync_status() == 0
    y_ref, L = orc_mt.gemm(xq, sx, wq, sw)
    assert_gemm_close(host(y), y_ref, L, f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (1, 1536, 7168),    # the decode shape: K over a cluster of 8 CTAs, 7 chunks each
    (33, 300, 1280),    # 10 chunks: clusters of 5 CTAs of 2 chunks; 48 token columns; ragged N
    (64, 256, 8192),    # 64 chunks: 8 per CTA (each in its own stage and TMEM columns), 64 tokens
    (16, 7168, 7168),   # 56 weight tiles x 8 CTAs: several waves of clusters
    (2, 1, 384),        # one output column, 3 chunks
    (128, 256, 512),    # the tiny configuration's shape: 128 token columns, one chunk per CTA
    (100, 300, 2048),   # 112 token columns (30 KB stages, 4 chunks at most): 2 chunks on each of 8 CTAs
    (128, 1536, 4096),  # 128 token columns, 4 chunks per CTA: all 512 TMEM columns
])
def test_gemm_few_tokens(F, orc, M, N, K):
    """Few tokens (M <= 128 and K within the cluster's chunk budget) take the
    weight-streaming kernel (weight rows on the MMA's 128-row side, tokens on
    N, K split over a cluster and summed through distributed shared memory):
    every element against the oracle, the same bits with and without a
    workspace, and run to run."""
    rng = np.random.default_rng(M + N + K)
    x = synth.activations(rng, M, K, n_outlier=4, outlier_scale=25.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    assert F.fp8bs_gemm_workspace_size(M, N, K) == 0
    _, y1 = _gemm_only(F, orc, x, w, workspace=True)
    _, y2 = _gemm_only(F, orc, x, w, workspace=False)
    assert np.array_equal(y1, y2)


@pytest.mark.parametrize("M,N,K", [(5, 300, 1024), (128, 200, 512)])
def test_gemm_strided_output(F, orc, M, N, K):
    """y as a column slice of a wider buffer (ldy > N): every element of the
    slice against the oracle, the columns outside it untouched.  Both shapes
    take the few-token kernel, whose reduction stores the output itself."""
    rng = np.random.default_rng(M + N)
    x = synth.activations(rng, M, K, n_outlier=2, outlier_scale=25.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    xq, sx = orc.act_quant(x, lds=max(4, (K // 128 + 3) // 4 * 4))
    wq, sw = orc.weight_quant(w)
    ld = (N + 72 + 7) // 8 * 8  # the row stride must be a multiple of 8 elements
    big = torch.full((M, ld), 7.0, dtype=torch.bfloat16, device="cuda")
    y = big[:, 40:40 + N]  # 80 bytes in: 16-byte aligned
    F.fp8bs_gemm(dev(xq), dev(sx), dev(wq), dev(sw), y=y)
    assert F.fp8bs_sync_status() == 0
    y_ref, L = orc.gemm(xq, sx, wq, sw)
    assert_gemm_close(host(y.contiguous()), y_ref, L, f"strided y {M}x{N}x{K}")
    rest = torch.cat([big[:, :40], big[:, 40 + N:]], dim=1)
    assert bool((rest == 7.0).all())


@pytest.mark.parametrize("M", [1, 16, 64, 96])
def test_gemm_decode_split_k_matches_unsplit(F, orc, M):
    """q_down (K = 7168): M <= 64 runs the weight-streaming kernel with or
    without a workspace; M = 96 (too many chunks for its 96 token columns)
    uses the split-K plan when a workspace is given.  Every plan is within the
    bound and bit-reproducible run to run."""
    c = synth.q_down(M)
    r1, y1 = _gemm_only(F, orc, c.x, c.w, workspace=True)
    r2, y2 = _gemm_only(F, orc, c.x, c.w, workspace=False)
    _, y3 = _gemm_only(F, orc, c.x, c.w, workspace=True)
    assert np.array_equal(y1, y3)


def test_gemm_deterministic(F, orc):
    c = synth.tiny()
    _, a = _gemm_only(F, orc, c.x, c.w)
    _, b = _gemm_only(F, orc, c.x, c.w)
    assert np.array_equal(a, b)


def test_gemm_identity_weight_exact(F, orc):
    """W = I: y = bf16(dec(xq) * sx * 448 * s_diag), i.e. the dequantised x
    scaled by 448*RN(1/448) -- checked against the oracle to the bound and the
    codes' sign/zero pattern exactly."""
    rng = np.random.default_rng(9)
    x = synth.activations(rng, 256, 512)
    w = synth.to_bf16_bits(np.eye(512, dtype=np.float32))
    _gemm_only(F, orc, x, w)


def _pipeline(F, orc, orc_mt, case, chunk=2048):
    """Device: weight_quant + act_quant + gemm (the bench's launch) vs the
    oracle's pipeline on the same bf16 inputs, every output element."""
    M, N, K = case.shape
    x = dev_bf16(case.x)
    w = dev_bf16(case.w)
    wq, sw = F.fp8bs_weight_quant(w)
    xq, sx = F.fp8bs_act_quant(x)
    n = F.fp8bs_gemm_workspace_size(M, N, K)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if n else None
    y = F.fp8bs_gemm(xq, sx, wq, sw, workspace=ws)
    assert F.fp8bs_sync_status() == 0
    yh = host(y)
    del x, w, wq, sw, xq, sx, y, ws
    wq_o, sw_o = orc.weight_quant(case.w)
    worst = 0.0
    for r0 in range(0, M, chunk):
        r1 = min(M, r0 + chunk)
        xq_o, sx_o = orc.act_quant(case.x[r0:r1])
        y_ref, L = orc_mt.gemm(xq_o, sx_o, wq_o, sw_o)
        worst = max(worst, assert_gemm_close(yh[r0:r1], y_ref, L, f"{case.name} rows {r0}..{r1 - 1}"))
    return worst


def test_pipeline_kv_down_full(F, orc, orc_mt):
    _pipeline(F, orc, orc_mt, synth.kv_down())


def test_stream_order_with_shared_buffers(F, orc):
    """Kernels start early under programmatic dependent launch; each must wait
    for its predecessor before touching memory.  Two inputs alternate through
    one Xq/Sx and one Wq/Sw buffer on one stream with no host sync between
    calls, so every weight_quant and act_quant overwrites what the GEMM just
    before it reads (write after read), and every GEMM reads what was just
    written (read after write).  Each output must match its own inputs."""
    c1 = synth.kv_down()
    M, N, K = c1.shape
    rng = np.random.default_rng(77)
    x2 = synth.activations(rng, M, K, n_outlier=16, outlier_scale=10.0)
    w2 = synth.normal_bf16(rng, (N, K), 0.05)
    cases = [(c1.x, c1.w), (x2, w2)]
    xs = [dev_bf16(x) for x, _ in cases]
    ws = [dev_bf16(w) for _, w in cases]
    lds = (K // 128 + 3) // 4 * 4
    xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty((M, lds), dtype=torch.float32, device="cuda")
    wq = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    ys = []
    for rep in range(3):
        for i in range(2):
            F.fp8bs_weight_quant(ws[i], wq=wq, sw=sw)
            F.fp8bs_act_quant(xs[i], xq=xq, sx=sx)
            ys.append((i, F.fp8bs_gemm(xq, sx, wq, sw)))
    assert F.fp8bs_sync_status() == 0
    rows = sample_rows(M, 16, seed=5)
    for i, (x, w) in enumerate(cases):
        xq_o, sx_o = orc.act_quant(x[rows])
        wq_o, sw_o = orc.weight_quant(w)
        y_ref, L = orc.gemm(xq_o, sx_o, wq_o, sw_o)
        outs = [host(y) for j, y in ys if j == i]
        assert_gemm_close(outs[0][rows], y_ref, L, f"input {i}")
        for o in outs[1:]:
            assert np.array_equal(o, outs[0]), f"input {i}: a repetition differs"


@pytest.mark.parametrize("M", list(synth.Q_SWEEP_M))
def test_pipeline_q_sweep_full(F, orc, orc_mt, M):
    _pipeline(F, orc, orc_mt, synth.q_down(M))


def test_pipeline_large_square_full(F, orc, orc_mt):
    _pipeline(F, orc, orc_mt, synth.large_square())
