"""GPU parity of fp8bs_grouped_gemm_swiglu: the MoE expert first stage,
h = silu(x w1^T) * (x w3^T) per expert (the pages' Expert forward before w2),
against the oracle's exact grouped GEMMs and fp64 silu.

Bound.  a and b are the exact GEMM outputs, ta and tb their GEMM bounds
(2^-8 |y| + 1e-4 L, which also covers rounding each to bf16).  silu has
slope at most 1.1, so |silu(a~) - silu(a)| <= 1.1 ta; silu's bf16 rounding
adds 2^-8 S (S = |silu(a)| + 1.1 ta bounds |silu(a~)|) and its fp32
evaluation a little more; the product's bf16 rounding adds 2^-8 of the
product.  Hence
  |h - silu(a) b| <= (1.1 ta + (2^-8 + 2^-20) S)(|b| + tb) + |silu(a)| tb
                     + 2^-8 (1 + 2^-8) S (|b| + tb).
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import dev, host
from oracle import gemm_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _case(orc, counts, I, K, seed):
    rng = np.random.default_rng(seed)
    G = len(counts)
    off = synth.offsets_from_counts(counts)
    T = int(off[-1])
    x = synth.activations(rng, T, K, n_outlier=min(8, K // 64), outlier_scale=10.0)
    xq, sx = orc.act_quant(x, lds=max(4, (K // 128 + 3) // 4 * 4))
    w1q, sw1, w3q, sw3 = [], [], [], []
    for _ in range(G):
        q, s = orc.weight_quant(synth.normal_bf16(rng, (I, K), 0.03))
        w1q.append(q); sw1.append(s)
        q, s = orc.weight_quant(synth.normal_bf16(rng, (I, K), 0.03))
        w3q.append(q); sw3.append(s)
    return xq, sx, np.stack(w1q), np.stack(sw1), np.stack(w3q), np.stack(sw3), off


def _bound(orc, xq, sx, w1q, sw1, w3q, sw3, off, rows):
    h_ref, a, b, La, Lb = orc.grouped_swiglu(xq, sx, w1q, sw1, w3q, sw3, off, rows=rows)
    ta, tb = gemm_tolerance(a, La), gemm_tolerance(b, Lb)
    s_abs = np.abs(orc.swiglu(a, np.ones_like(a)))
    S = s_abs + 1.1 * ta
    B = np.abs(b) + tb
    bound = (1.1 * ta + (2.0 ** -8 + 2.0 ** -20) * S) * B + s_abs * tb + 2.0 ** -8 * (1 + 2.0 ** -8) * S * B
    return h_ref, bound


def _check(orc, h, xq, sx, w1q, sw1, w3q, sw3, off, rows, what):
    h_ref, bound = _bound(orc, xq, sx, w1q, sw1, w3q, sw3, off, rows)
    hf = (host(h)[rows].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bad = np.abs(hf - h_ref) > bound + 1e-30
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside the bound"
    # the bound is not vacuous: most outputs sit far inside it
    assert np.median(np.abs(hf - h_ref) / (bound + 1e-30)) < 0.5


def test_swiglu_small_all_rows(F, orc):
    """Five experts: ragged row counts, an empty expert, a one-row expert."""
    counts = [3, 0, 130, 1, 40]
    xq, sx, w1q, sw1, w3q, sw3, off = _case(orc, counts, I=256, K=384, seed=41)
    h = F.fp8bs_grouped_gemm_swiglu(dev(xq), dev(sx), dev(w1q), dev(sw1), dev(w3q), dev(sw3),
                                    torch.from_numpy(off).cuda())
    assert F.fp8bs_sync_status() == 0
    _check(orc, h, xq, sx, w1q, sw1, w3q, sw3, off, np.arange(off[-1]), "swiglu small")


def test_swiglu_wider(F, orc):
    """Four experts with several h tiles (I = 512) and 16 K chunks."""
    counts = [200, 1, 129, 77]
    xq, sx, w1q, sw1, w3q, sw3, off = _case(orc, counts, I=512, K=2048, seed=42)
    h = F.fp8bs_grouped_gemm_swiglu(dev(xq), dev(sx), dev(w1q), dev(sw1), dev(w3q), dev(sw3),
                                    torch.from_numpy(off).cuda())
    assert F.fp8bs_sync_status() == 0
    rng = np.random.default_rng(3)
    rows = np.union1d(np.array([0, 199, 200, 201, 329, 330, 406]), rng.choice(int(off[-1]), 60, replace=False))
    _check(orc, h, xq, sx, w1q, sw1, w3q, sw3, off, rows, "swiglu wider")


def test_swiglu_matches_two_grouped_gemms(F, orc):
    """The fused call against the library's own two grouped GEMMs followed by
    the same bf16 arithmetic on the host: the GEMM halves are the same kernel
    pipeline, so a and b agree bit for bit before the activation."""
    counts = [65, 0, 130]
    xq, sx, w1q, sw1, w3q, sw3, off = _case(orc, counts, I=256, K=512, seed=43)
    d = [dev(t) for t in (xq, sx, w1q, sw1, w3q, sw3)]
    offd = torch.from_numpy(off).cuda()
    h = F.fp8bs_grouped_gemm_swiglu(*d, offd)
    a = F.fp8bs_grouped_gemm(d[0], d[1], d[2], d[3], offd)
    b = F.fp8bs_grouped_gemm(d[0], d[1], d[4], d[5], offd)
    assert F.fp8bs_sync_status() == 0
    af, bf = a.float(), b.float()
    sg = (af / (1.0 + torch.exp(-af))).to(torch.bfloat16).float()
    h_host = (sg * bf).to(torch.bfloat16)
    hh, hr = host(h), host(h_host)
    # silu's fp32 evaluation may differ in the last bit between torch and the
    # kernel; the bf16 result then differs by at most one bf16 step
    diff = np.abs(hh.astype(np.int32) - hr.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99


@pytest.mark.parametrize("counts,I,K", [([3, 0, 130, 1, 40], 256, 384), ([200, 1, 129, 77], 512, 1024)])
def test_swiglu_fp8_out(F, orc, counts, I, K):
    """h quantised in the same pass (a row's 128-column group spans both
    promotion warpgroups): bit-identical to act_quant of the bf16 h, the same
    without h, and within the bound plus half an e4m3 step of the oracle."""
    import ml_dtypes
    xq, sx, w1q, sw1, w3q, sw3, off = _case(orc, counts, I=I, K=K, seed=44 + I)
    d = [dev(t) for t in (xq, sx, w1q, sw1, w3q, sw3)]
    offd = torch.from_numpy(off).cuda()
    h, hq, sh = F.fp8bs_grouped_gemm_swiglu(*d, offd, want_fp8=True)
    _, hq2, sh2 = F.fp8bs_grouped_gemm_swiglu(*d, offd, want_h=False, want_fp8=True)
    xq2, sx2 = F.fp8bs_act_quant(h)
    assert F.fp8bs_sync_status() == 0
    hq_h, sh_h = host(hq), host(sh)
    assert np.array_equal(hq_h, host(xq2))
    assert np.array_equal(sh_h.view(np.uint32), host(sx2)[:, : I // 128].view(np.uint32))
    assert np.array_equal(host(hq2), hq_h)
    assert np.array_equal(host(sh2).view(np.uint32), sh_h.view(np.uint32))
    rows = np.arange(off[-1])
    h_ref, bound = _bound(orc, xq, sx, w1q, sw1, w3q, sw3, off, rows)
    v = np.arange(256, dtype=np.uint8).view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    s = np.repeat(sh_h.astype(np.float64), 128, axis=1)
    deq = v[hq_h] * s
    full = bound + np.ldexp(np.abs(h_ref) + bound, -4) * (1 + 2.0 ** -20) + np.ldexp(s, -10) + 1e-30
    bad = np.abs(deq - h_ref) > full
    assert not bad.any(), f"{int(bad.sum())} fp8 h outside the bound"
