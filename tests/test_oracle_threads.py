"""The oracle's OpenMP build (liboracle_omp.so, used by the full-size parity
tests) is the same source as the pinned single-threaded build: its GEMM and
grouped GEMM must return the same fp64 values bit for bit."""
import numpy as np

from fp8_block_scaled_18_b300 import synth


def test_threaded_gemm_equals_single_threaded(orc, orc_mt):
    rng = np.random.default_rng(11)
    M, N, K = 77, 300, 640
    x = synth.activations(rng, M, K, n_outlier=6, outlier_scale=30.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    xq, sx = orc.act_quant(x, lds=8)
    wq, sw = orc.weight_quant(w)
    rows = rng.permutation(M)[:50]
    for r in (None, rows):
        y1, L1 = orc.gemm(xq, sx, wq, sw, rows=r)
        y2, L2 = orc_mt.gemm(xq, sx, wq, sw, rows=r)
        assert np.array_equal(y1.view(np.uint64), y2.view(np.uint64))
        assert np.array_equal(L1.view(np.uint64), L2.view(np.uint64))


def test_threaded_grouped_equals_single_threaded(orc, orc_mt):
    rng = np.random.default_rng(12)
    counts = np.array([5, 0, 40, 1, 0, 33])
    off = synth.offsets_from_counts(counts)
    T, N, K = int(off[-1]), 136, 256
    x = synth.activations(rng, T, K)
    w = synth.normal_bf16(rng, (counts.size, N, K), 0.02)
    xq, sx = orc.act_quant(x)
    wqs, sws = zip(*[orc.weight_quant(w[g]) for g in range(counts.size)])
    wq, sw = np.stack(wqs), np.stack(sws)
    rows = rng.permutation(T)  # listed out of order, experts interleaved
    y1, L1 = orc.grouped_gemm(xq, sx, wq, sw, off, rows=rows)
    y2, L2 = orc_mt.grouped_gemm(xq, sx, wq, sw, off, rows=rows)
    assert np.array_equal(y1.view(np.uint64), y2.view(np.uint64))
    assert np.array_equal(L1.view(np.uint64), L2.view(np.uint64))
    # each row equals the dense product with its own expert's weight
    for g in range(counts.size):
        r0, r1 = int(off[g]), int(off[g + 1])
        if r1 > r0:
            yd, _ = orc.gemm(xq[r0:r1], sx[r0:r1], wq[g], sw[g])
            pos = np.nonzero((rows >= r0) & (rows < r1))[0]
            assert np.array_equal(y1[pos], yd[rows[pos] - r0])


def test_threaded_wgrad_equals_single_threaded(orc, orc_mt):
    rng = np.random.default_rng(13)
    M, N, K = 300, 136, 256   # a ragged last block of tokens
    dy = synth.activations(rng, M, N, n_outlier=3, outlier_scale=10.0)
    x = synth.activations(rng, M, K)
    dyq, sdy = orc.act_quant_cols(dy)
    xq, sx = orc.act_quant_cols(x)
    dw1, L1 = orc.gemm_wgrad(dyq, sdy, xq, sx)
    rows = np.array([5, 0, 135, 64], dtype=np.int64)
    dw2, L2 = orc_mt.gemm_wgrad(dyq, sdy, xq, sx, rows=rows)
    assert np.array_equal(dw2.view(np.uint64), dw1[rows].view(np.uint64))
    assert np.array_equal(L2.view(np.uint64), L1[rows].view(np.uint64))
