"""Pins that tie the CPU oracle to facts fixed outside itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  tests/test_oracle_pins.py runs them on the real oracle;
tests/test_oracle_mutants.py runs them on copies of the oracle with a planted
mistake and requires every mistake to be caught by at least one pin.

The expected values come from: exact rational arithmetic (fractions), closed
forms that hold by construction (power-of-two scales, e4m3-representable
operands), integer arithmetic, and independent libraries (ml_dtypes, numpy).
"""
from __future__ import annotations

from fractions import Fraction

import ml_dtypes
import numpy as np

from fp8_block_scaled_18_b300 import synth

E4M3_MAX = 448

# ---------------------------------------------------------------------------
# exact helpers (independent of the oracle's C code)
# ---------------------------------------------------------------------------


def f32_round(fr: Fraction) -> float:
    """Round an exact rational to the nearest binary32 value, ties to even."""
    if fr == 0:
        return 0.0
    neg = fr < 0
    a = -fr if neg else fr
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    e = max(e, -126)
    scaled = a / Fraction(2) ** (e - 23)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = Fraction(n) * Fraction(2) ** (e - 23)
    if val >= Fraction(2) ** 128:
        out = float("inf")
    else:
        out = float(val)  # exact: n has <= 24 bits
    return -out if neg else out


def e4m3_values() -> np.ndarray:
    """All 254 finite e4m3 values indexed by code (NaN codes -> nan), from ml_dtypes."""
    return np.arange(256, dtype=np.uint8).view(ml_dtypes.float8_e4m3fn).astype(np.float64)


def e4m3_code_lib(v: np.ndarray) -> np.ndarray:
    """Library encode with saturation: clip to +-448 then ml_dtypes RNE cast."""
    v = np.clip(np.asarray(v, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    return v.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)


def bf16_bits(v) -> np.ndarray:
    return synth.to_bf16_bits(np.asarray(v, dtype=np.float32))


def f32_of_bf16(bits) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits)


def _pos_codes_with_max(rng, n, allow_sub=True):
    """n positive-or-negative e4m3 codes with |max| == 448 (code 0x7E present)."""
    lo = 0 if allow_sub else 0x08
    mags = rng.integers(lo, 0x7E, size=n)            # 0 .. 447-ish, excludes NaN
    signs = rng.integers(0, 2, size=n) * 0x80
    codes = (mags | signs).astype(np.uint8)
    codes[rng.integers(0, n)] = 0x7E | (0x80 if rng.integers(0, 2) else 0)
    return codes


# ---------------------------------------------------------------------------
# codec
# ---------------------------------------------------------------------------


def pin_codec_midpoints(o):
    pos = [c for c in range(0x7F)]
    vals = e4m3_values()[pos]
    mids, want = [], []
    for i in range(len(pos) - 1):
        mid = (vals[i] + vals[i + 1]) / 2
        mids.append(mid)
        want.append(pos[i] if pos[i] % 2 == 0 else pos[i + 1])
    got = o.e4m3_encode(np.array(mids, dtype=np.float32))
    assert np.array_equal(got, np.array(want, dtype=np.uint8)), "midpoint ties must go to the even code"


# ---------------------------------------------------------------------------
# act_quant
# ---------------------------------------------------------------------------


def pin_act_quant_rank1(o):
    """x[m,k] = 2^a_m * c_k with each 128-group of c holding a +-448: then
    s = 2^a_m exactly and the codes are c's codes exactly."""
    rng = np.random.default_rng(11)
    M, K = 24, 512
    codes = np.concatenate([_pos_codes_with_max(rng, 128) for _ in range(K // 128)])
    c = e4m3_values()[codes]
    a = rng.integers(-20, 20, size=M)
    x = np.ldexp(c[None, :], a[:, None])
    xb = bf16_bits(x)
    assert np.array_equal(f32_of_bf16(xb).astype(np.float64), x)  # exactly representable
    xq, sx = o.act_quant(xb)
    assert np.array_equal(sx, np.ldexp(np.ones((M, K // 128), np.float32), a[:, None]).astype(np.float32))
    assert np.array_equal(xq, np.broadcast_to(codes, (M, K)))


def _division_sensitive_groups(rng, n_groups):
    """Groups [amax, x, x, ...] whose quotient x/s lies within a few fp32 ulps
    of an e4m3 rounding boundary, where dividing and multiplying by a rounded
    reciprocal can disagree.  Found by a numpy search (inputs only)."""
    xs = f32_of_bf16(np.arange(0x3C00, 0x4400, dtype=np.uint16))  # bf16 in [2^-7, 2^8)
    groups = []
    tries = 0
    while len(groups) < n_groups and tries < 4000:
        tries += 1
        amax = np.float32(f32_of_bf16(np.array([rng.integers(0x4000, 0x4300)], np.uint16))[0])
        s = np.float32(amax / np.float32(448))
        cand = xs[xs < amax]
        q_div = cand / s
        q_mul = cand * np.float32(np.float32(448) / amax)
        diff = e4m3_code_lib(q_div) != e4m3_code_lib(q_mul)
        if diff.any():
            pick = cand[diff][:127]
            g = np.full(128, pick[0], np.float32)
            g[0] = amax
            g[1:1 + pick.size] = pick
            groups.append(g)
    assert len(groups) == n_groups, "search for division-sensitive inputs failed"
    return np.stack(groups)


def pin_act_quant_division_exact(o):
    """Brute force in exact rationals: s = RN32(amax/448), q = e4m3(RN32(x/s))."""
    rng = np.random.default_rng(12)
    rnd = rng.standard_normal((6, 128)).astype(np.float32) * np.float32(3)
    rnd[2] *= np.float32(1e-30)                 # tiny values, fp32 subnormal quotients
    rnd[3, :] = 0
    rnd[3, 5] = -1.5                            # single nonzero
    groups = np.concatenate([rnd, _division_sensitive_groups(rng, 6)])
    xb = bf16_bits(groups).reshape(1, -1)
    xq, sx = o.act_quant(xb)
    xf = f32_of_bf16(xb).reshape(groups.shape)
    for g in range(groups.shape[0]):
        amax = max(Fraction(float(abs(v))) for v in xf[g])
        s = f32_round(amax / 448)
        assert sx[0, g] == np.float32(s), (g, sx[0, g], s)
        want = []
        for v in xf[g]:
            if amax == 0:
                want.append(0x80 if np.signbit(v) else 0)
            else:
                want.append(int(e4m3_code_lib(np.float32(f32_round(Fraction(float(v)) / Fraction(s))))))
        got = xq[0, g * 128:(g + 1) * 128]
        assert np.array_equal(got, np.array(want, np.uint8)), (g, np.nonzero(got != np.array(want))[0][:5])


def pin_act_quant_invariants(o):
    rng = np.random.default_rng(13)
    M, K = 16, 1024
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(2.0)
    x[3, 128:256] = 0.0                          # zero group
    x[4, 256:384] = -0.0                         # negative-zero group
    x[5, :128] = np.float32(1e-3) * x[5, :128]   # small group
    xb = bf16_bits(x)
    xq, sx = o.act_quant(xb)
    xf = f32_of_bf16(xb)
    dec = e4m3_values()[xq]
    for m in range(M):
        for g in range(K // 128):
            sl = slice(g * 128, (g + 1) * 128)
            grp, q, s = xf[m, sl], xq[m, sl], sx[m, g]
            if not np.any(grp):
                assert s == 0 and np.array_equal(q, np.where(np.signbit(grp), 0x80, 0).astype(np.uint8))
                continue
            assert s > 0 and (q & 0x7F).max() == 0x7E          # the amax element maps to 448
            err = np.abs(grp.astype(np.float64) - dec[m, sl] * float(s))
            bound = np.maximum(np.abs(grp) * 2.0 ** -4, float(s) * 2.0 ** -10)
            assert np.all(err <= bound)
            assert np.array_equal(q & 0x80, np.where(np.signbit(grp), 0x80, 0).astype(np.uint8))
    # sign symmetry and power-of-two scaling
    xq2, sx2 = o.act_quant(bf16_bits(-xf))
    assert np.array_equal(sx2, sx) and np.array_equal(xq2 ^ 0x80, xq)
    xq3, sx3 = o.act_quant(bf16_bits(xf * np.float32(2.0 ** 7)))
    assert np.array_equal(sx3, sx * np.float32(2.0 ** 7)) and np.array_equal(xq3, xq)
    # quantising gathered rows == gathering quantised rows
    perm = rng.permutation(M)
    xq4, sx4 = o.act_quant(xb[perm])
    assert np.array_equal(xq4, xq[perm]) and np.array_equal(sx4, sx[perm])


# ---------------------------------------------------------------------------
# weight_quant / weight_dequant
# ---------------------------------------------------------------------------


def _block_closed_form(rng, N, K):
    """w = 2^b[nb,kb] * d with each 128x128 block of d holding a +-448 in its
    valid rows: s = 2^b and codes = d's codes, exactly."""
    NB, KB = (N + 127) // 128, K // 128
    codes = (rng.integers(0, 0x7E, size=(N, K)) | (rng.integers(0, 2, size=(N, K)) * 0x80)).astype(np.uint8)
    b = rng.integers(-12, 6, size=(NB, KB))
    for nb in range(NB):
        for kb in range(KB):
            r = rng.integers(nb * 128, min(N, nb * 128 + 128))
            codes[r, kb * 128 + rng.integers(0, 128)] = 0x7E
    scale = np.ldexp(np.ones((N, K)), np.repeat(np.repeat(b, 128, 0)[:N], 128, 1))
    w = e4m3_values()[codes] * scale
    return codes, b, w


def pin_weight_quant_blocks(o):
    rng = np.random.default_rng(14)
    for N, K in ((256, 384), (576, 256), (130, 128)):
        codes, b, w = _block_closed_form(rng, N, K)
        wb = bf16_bits(w)
        assert np.array_equal(f32_of_bf16(wb).astype(np.float64), w)
        wq, sw = o.weight_quant(wb)
        assert np.array_equal(sw, np.ldexp(np.ones(b.shape, np.float32), b).astype(np.float32)), (N, K)
        assert np.array_equal(wq, codes), (N, K)


def pin_weight_quant_identity(o):
    """W = I (512x512): diagonal blocks s = RN32(1/448) with the diagonal at
    code 0x7E; every other entry code 0 and off-diagonal blocks s = 0."""
    w = bf16_bits(np.eye(512, dtype=np.float32))
    wq, sw = o.weight_quant(w)
    s_diag = np.float32(f32_round(Fraction(1, 448)))
    assert np.array_equal(sw, np.where(np.eye(4, dtype=bool), s_diag, np.float32(0)))
    assert np.array_equal(wq, np.where(np.eye(512, dtype=bool), 0x7E, 0).astype(np.uint8))


def pin_weight_quant_ragged(o):
    """N = 576: five row blocks; the last uses its 64 valid rows, which gives
    the same codes and scales as zero-padding the weight to 640 rows."""
    rng = np.random.default_rng(15)
    w = bf16_bits(rng.standard_normal((576, 256)).astype(np.float32) * np.float32(0.02))
    wq, sw = o.weight_quant(w)
    assert sw.shape == (5, 2)
    wpad = np.zeros((640, 256), np.uint16)
    wpad[:576] = w
    wq2, sw2 = o.weight_quant(wpad)
    assert np.array_equal(sw, sw2) and np.array_equal(wq, wq2[:576]) and not np.any(wq2[576:])
    wf = f32_of_bf16(w)
    assert sw[4, 1] == np.float32(f32_round(Fraction(float(np.abs(wf[512:, 128:]).max())) / 448))


def pin_weight_dequant(o):
    rng = np.random.default_rng(16)
    codes, b, w = _block_closed_form(rng, 256, 256)
    sw = np.ldexp(np.ones(b.shape, np.float32), b).astype(np.float32)
    back = o.weight_dequant(codes, sw)
    assert np.array_equal(f32_of_bf16(back).astype(np.float64), w)   # exact for power-of-two scales
    # general scales: one fp32 rounding of the exact product, then bf16 RNE
    sw2 = (rng.uniform(0.5, 2.0, size=(2, 2)) * 1e-3).astype(np.float32)
    back2 = o.weight_dequant(codes, sw2)
    dec = e4m3_values()[codes]
    s_full = np.repeat(np.repeat(sw2, 128, 0), 128, 1)
    for (n, k) in zip(rng.integers(0, 256, 300), rng.integers(0, 256, 300)):
        p = f32_round(Fraction(float(dec[n, k])) * Fraction(float(s_full[n, k])))
        want = synth.to_bf16_bits(np.array([p], np.float32))[0]
        assert back2[n, k] == want, (n, k)
    # quantise -> dequantise stays within e4m3's relative step
    wr = bf16_bits(rng.standard_normal((256, 256)).astype(np.float32) * np.float32(0.02))
    wq, swr = o.weight_quant(wr)
    wr2 = f32_of_bf16(o.weight_dequant(wq, swr)).astype(np.float64)
    x = f32_of_bf16(wr).astype(np.float64)
    s_full = np.repeat(np.repeat(swr, 128, 0), 128, 1).astype(np.float64)
    assert np.all(np.abs(wr2 - x) <= np.maximum(np.abs(x) * (2.0 ** -4 + 2.0 ** -8), s_full * 2.0 ** -9))


# ---------------------------------------------------------------------------
# gemm
# ---------------------------------------------------------------------------


def _exact_gemm(xq, sx, wq, sw, m, n):
    vals = e4m3_values()
    K = xq.shape[1]
    tot = Fraction(0)
    for kb in range(K // 128):
        bsum = Fraction(0)
        for k in range(kb * 128, (kb + 1) * 128):
            bsum += Fraction(float(vals[xq[m, k]])) * Fraction(float(vals[wq[n, k]]))
        tot += Fraction(float(sx[m, kb])) * Fraction(float(sw[n // 128, kb])) * bsum
    return tot


def pin_gemm_bruteforce(o):
    """Tiny shapes against exact rational arithmetic."""
    rng = np.random.default_rng(17)
    for (M, N, K) in ((3, 5, 128), (4, 130, 256), (2, 3, 384)):
        xq = rng.integers(0, 0xFF, size=(M, K)).astype(np.uint8)
        xq[(xq & 0x7F) == 0x7F] = 0x7E
        wq = rng.integers(0, 0xFF, size=(N, K)).astype(np.uint8)
        wq[(wq & 0x7F) == 0x7F] = 0x7E
        sx = rng.uniform(1e-3, 1.0, size=(M, K // 128)).astype(np.float32)
        sw = rng.uniform(1e-4, 1e-2, size=((N + 127) // 128, K // 128)).astype(np.float32)
        y, L = o.gemm(xq, sx, wq, sw)
        for m in range(M):
            for n in list(range(min(N, 6))) + [N - 1]:
                ex = _exact_gemm(xq, sx, wq, sw, m, n)
                assert abs(Fraction(float(y[m, n])) - ex) <= Fraction(2) ** -45 * Fraction(float(L[m, n])) + Fraction(1, 10 ** 300), (M, N, K, m, n)


def pin_gemm_rank1(o):
    """Full path on closed-form inputs: x = 2^a_m c_k, w = 2^b_(n,kb) d_(n,k)
    quantise losslessly, so y = sum_k 2^(a_m + b) c_k d_(n,k), in integers."""
    rng = np.random.default_rng(18)
    M, N, K = 8, 256, 384
    ccodes = np.concatenate([_pos_codes_with_max(rng, 128) for _ in range(K // 128)])
    a = rng.integers(-6, 6, size=M)
    x = np.ldexp(e4m3_values()[ccodes][None, :], a[:, None])
    dcodes, b, w = _block_closed_form(rng, N, K)
    xq, sx = o.act_quant(bf16_bits(x))
    wq, sw = o.weight_quant(bf16_bits(w))
    y, L = o.gemm(xq, sx, wq, sw)
    ci = (e4m3_values()[ccodes] * 512).astype(np.int64)          # e4m3 values are multiples of 2^-9
    di = (e4m3_values()[dcodes] * 512).astype(np.int64)
    for m in range(M):
        for n in range(0, N, 17):
            ex = Fraction(0)
            for kb in range(K // 128):
                sl = slice(kb * 128, (kb + 1) * 128)
                ex += Fraction(int(np.dot(ci[sl], di[n, sl]))) * Fraction(2) ** int(a[m] + b[n // 128, kb] - 18)
            assert Fraction(float(y[m, n])) == ex, (m, n)


def pin_gemm_diag(o):
    """W = diag(d) with e4m3 codes, power-of-two block scales:
    y[m,n] = dec(xq[m,n]) sx[m,n/128] dec(d_n) sw[n/128,n/128], exactly."""
    rng = np.random.default_rng(19)
    M, K = 5, 256
    xq = rng.integers(0, 0x7E, size=(M, K)).astype(np.uint8) | (rng.integers(0, 2, (M, K)) * 0x80).astype(np.uint8)
    sx = rng.uniform(0.1, 10, size=(M, 2)).astype(np.float32)
    d = rng.integers(0x30, 0x50, size=K).astype(np.uint8)
    wq = np.zeros((K, K), np.uint8)
    wq[np.arange(K), np.arange(K)] = d
    sw = np.ldexp(np.ones((2, 2), np.float32), rng.integers(-3, 3, size=(2, 2))).astype(np.float32)
    y, _ = o.gemm(xq, sx, wq, sw)
    v = e4m3_values()
    for m in range(M):
        for n in range(K):
            want = Fraction(float(v[xq[m, n]])) * Fraction(float(sx[m, n // 128])) * \
                Fraction(float(v[d[n]])) * Fraction(float(sw[n // 128, n // 128]))
            assert Fraction(float(y[m, n])) == want, (m, n)


def pin_gemm_vs_dequant_matmul(o):
    """The bf16 branch of linear(): dequantise both operands, one matmul."""
    rng = np.random.default_rng(20)
    case = synth.tiny(0)
    xq, sx = o.act_quant(case.x)
    wq, sw = o.weight_quant(case.w)
    v = e4m3_values()
    xd = v[xq] * np.repeat(sx.astype(np.float64), 128, 1)
    wd = v[wq] * np.repeat(np.repeat(sw.astype(np.float64), 128, 0), 128, 1)[: wq.shape[0]]
    ref = xd @ wd.T
    y, L = o.gemm(xq, sx, wq, sw)
    assert np.all(np.abs(y - ref) <= 1e-12 * L + 1e-300)
    rows = rng.choice(xq.shape[0], 7, replace=False)
    y2, _ = o.gemm(xq, sx, wq, sw, rows=rows)
    assert np.array_equal(y2, y[rows])


def pin_grouped(o):
    """Grouped = the dense product per expert over its row range; empty
    experts take no rows."""
    rng = np.random.default_rng(21)
    G, N, K = 5, 192, 256
    counts = np.array([3, 0, 7, 1, 0])
    off = synth.offsets_from_counts(counts)
    T = int(off[-1])
    xq = rng.integers(0, 0x7E, size=(T, K)).astype(np.uint8)
    sx = rng.uniform(0.1, 1.0, size=(T, K // 128)).astype(np.float32)
    wq = rng.integers(0, 0x7E, size=(G, N, K)).astype(np.uint8)
    sw = rng.uniform(1e-3, 1e-2, size=(G, 2, K // 128)).astype(np.float32)
    y, L = o.grouped_gemm(xq, sx, wq, sw, off)
    for g in range(G):
        r0, r1 = off[g], off[g + 1]
        if r1 > r0:
            yg, Lg = o.gemm(xq[r0:r1], sx[r0:r1], wq[g], sw[g])
            assert np.array_equal(y[r0:r1], yg) and np.array_equal(L[r0:r1], Lg)
    # one element against exact rationals
    m, n = 5, 150
    g = int(np.searchsorted(off, m, side="right") - 1)
    ex = _exact_gemm(xq[off[g]:off[g + 1]], sx[off[g]:off[g + 1]], wq[g], sw[g], m - off[g], n)
    assert abs(Fraction(float(y[m, n])) - ex) <= Fraction(2) ** -45 * Fraction(float(L[m, n]))


def pin_gemm_bias(o):
    """linear()'s bias: with an all-zero weight the output is the bias
    exactly; otherwise adding the bias changes each output by the bias's bf16
    value (fp64, up to one rounding of the sum)."""
    rng = np.random.default_rng(22)
    case = synth.tiny(0)
    N = case.w.shape[0]
    bias = synth.normal_bf16(rng, (N,), 1.0)
    bias_f = f32_of_bf16(bias).astype(np.float64)
    xq, sx = o.act_quant(case.x)
    wq0, sw0 = o.weight_quant(np.zeros_like(case.w))
    y0, _ = o.gemm(xq, sx, wq0, sw0, bias=bias)
    assert np.array_equal(y0, np.broadcast_to(bias_f, y0.shape))
    wq, sw = o.weight_quant(case.w)
    y, _ = o.gemm(xq, sx, wq, sw)
    yb, _ = o.gemm(xq, sx, wq, sw, bias=bias)
    assert np.all(np.abs((yb - y) - bias_f) <= 2.0 ** -52 * (np.abs(y) + np.abs(bias_f)))


def pin_swiglu(o):
    """The expert activation h = silu(a) * b against scipy's logistic
    function (silu(v) = v * expit(v)), its zero, its linear tail for large
    v and its vanishing tail for very negative v."""
    from scipy.special import expit
    rng = np.random.default_rng(23)
    a = np.concatenate([rng.standard_normal(1000) * 4, [0.0, 1.0, -1.0, 20.0, 40.0, -40.0]])
    b = rng.standard_normal(a.size)
    h = o.swiglu(a, b)
    assert np.allclose(h, a * expit(a) * b, rtol=1e-14, atol=1e-300)
    assert o.swiglu(np.array([0.0]), np.array([3.0]))[0] == 0.0
    assert abs(o.swiglu(np.array([40.0]), np.array([1.0]))[0] - 40.0) < 1e-12
    assert abs(o.swiglu(np.array([-40.0]), np.array([1.0]))[0]) < 1e-15


def pin_moe_dispatch(o):
    """Dispatch is a row gather: each routed row equals its token's codes and
    scales (numpy fancy indexing), and -- because the quantisation is per
    token row -- dispatching act_quant(x) equals act_quant of the gathered
    bf16 rows, bit for bit.  An out-of-range id gives a zero row."""
    case = synth.moe(seed=5, tokens=48, n_experts=16, n=256, k=384)
    xq, sx = o.act_quant(case.x_tokens)
    xr, sr = o.moe_dispatch(xq, sx, case.token_of_row)
    assert np.array_equal(xr, xq[case.token_of_row])
    assert np.array_equal(sr.view(np.uint32), sx[case.token_of_row, :3].view(np.uint32))
    xq2, sx2 = o.act_quant(case.x_rows)
    assert np.array_equal(xr, xq2) and np.array_equal(sr.view(np.uint32), sx2[:, :3].view(np.uint32))
    bad = np.array([2, -1, 48, 0], dtype=np.int32)
    xb, sb = o.moe_dispatch(xq, sx, bad)
    assert not xb[1:3].any() and not sb[1:3].any()
    assert np.array_equal(xb[[0, 3]], xq[[2, 0]])


def _combine_matrix(rows_of_token, w, R):
    """The combine as a [tokens, R] scatter matrix S (S[t, r_k] = w[r_k])."""
    tokens, topk = rows_of_token.shape
    S = np.zeros((tokens, R))
    np.add.at(S, (np.repeat(np.arange(tokens), topk), rows_of_token.reshape(-1)),
              w[rows_of_token.reshape(-1)].astype(np.float64))
    return S


def pin_moe_combine(o):
    """Combine = S @ Yk + z with the scatter matrix of the routing (numpy
    matmul, a different formulation of the same sum); with every expert
    output row equal to one vector c and gates that sum to 2.5 per token
    (the route_scale), y = 2.5 c + z exactly; with one routed expert of gate 1,
    y = that expert's row + z exactly."""
    case = synth.moe(seed=6, tokens=40, n_experts=32, n=256, k=256)
    R = case.token_of_row.size
    rng = np.random.default_rng(24)
    dim = 96
    yk = f32_of_bf16(synth.normal_bf16(rng, (R, dim), 1.0)).astype(np.float64)
    z = f32_of_bf16(synth.normal_bf16(rng, (40, dim), 1.0)).astype(np.float64)
    y, L = o.moe_combine(yk, case.weight_of_row, case.rows_of_token, z=z)
    ref = _combine_matrix(case.rows_of_token, case.weight_of_row, R) @ yk + z
    assert np.all(np.abs(y - ref) <= 1e-13 * L)
    assert np.all(L >= np.abs(y) * (1 - 1e-12))
    # closed form: gates 1.25, 0.5, 0.5, 0.25 (sum 2.5, exact), rows all c
    tokens, topk = 6, 4
    rt = np.arange(tokens * topk, dtype=np.int32).reshape(tokens, topk)[:, ::-1].copy()
    w = np.tile(np.array([0.25, 0.5, 0.5, 1.25], dtype=np.float32), tokens)
    c = f32_of_bf16(synth.normal_bf16(rng, (dim,), 1.0)).astype(np.float64)
    y2, _ = o.moe_combine(np.tile(c, (tokens * topk, 1)), w, rt)
    assert np.array_equal(y2, np.tile(2.5 * c, (tokens, 1)))
    # top-1 with gate 1: the expert row itself, plus z
    rt1 = rng.permutation(R)[:40].astype(np.int32).reshape(40, 1)
    y3, _ = o.moe_combine(yk, np.ones(R, dtype=np.float32), rt1, z=z)
    assert np.array_equal(y3, yk[rt1[:, 0]] + z)


def _gate_case(logits, dim=64):
    """x [T, dim], wg [E, dim] in bf16 with x . wg_e equal to the given
    (bf16-representable) logits exactly: x_t = the unit vector e_t-ish
    encoding, built as x[t] = one-hot of t (T <= dim) and wg[e, t] = logit."""
    T, E = logits.shape
    assert T <= dim
    x = np.zeros((T, dim), dtype=np.float32)
    x[np.arange(T), np.arange(T)] = 1.0
    wg = np.zeros((E, dim), dtype=np.float32)
    wg[:, :T] = logits.T
    return bf16_bits(x), bf16_bits(wg)


def pin_moe_gate(o):
    """Router, constructed cases whose answer is fixed by design: logits
    placed exactly (one-hot tokens), affinities against scipy's logistic
    function; the best groups are kept and an expert outside them is not
    chosen even when its score is higher than a chosen one; the bias moves the
    selection but not the gate values; the gate values are the chosen
    affinities normalised to 2.5."""
    from scipy.special import expit
    E, G = 16, 4                                   # 4 groups of 4 experts, keep 2, top-3
    lg = np.full((2, E), -4.0, dtype=np.float32)
    # token 0: group 0 = {0.5, 3, -1, 0.25}, group 1 = {2, 1.5, 1.75, 0}, group 2 = {2.5, -2, -2, -2}, group 3 low
    lg[0, :12] = [0.5, 3.0, -1.0, 0.25, 2.0, 1.5, 1.75, 0.0, 2.5, -2.0, -2.0, -2.0]
    # token 1: same, but the bias lifts expert 15 (group 3) to the top
    lg[1] = lg[0]
    x, wg = _gate_case(lg)
    bias = np.zeros(E, dtype=np.float32)
    ids, w, s = o.moe_gate(x, wg, bias, n_groups=G, topk_groups=2, top_k=3, want_scores=True)
    assert np.allclose(s, expit(lg.astype(np.float64)), rtol=1e-15, atol=0)
    # group maxima: g0 3.0, g2 2.5, g1 2.0 -> keep g0, g2; top-3 of {0.5,3,-1,.25,2.5,-2,-2,-2} = 1, 8, 0
    assert ids[0].tolist() == [1, 8, 0]
    # expert 4 (logit 2.0 > 0.5) is not chosen: its group is not kept
    ref = expit(np.array([3.0, 2.5, 0.5]))
    assert np.allclose(w[0], ref / ref.sum() * 2.5, rtol=1e-14)
    assert abs(w[0].sum() - 2.5) < 1e-14
    bias[15] = 0.99                                  # affinity expit(-4) = 0.018 + 0.99: top of group 3
    ids_b, w_b = o.moe_gate(x, wg, bias, n_groups=G, topk_groups=2, top_k=3)
    # group 3 (1.008) now outranks group 2 (0.924), which drops out with expert 8
    assert ids_b[1].tolist() == [15, 1, 0]
    ref_b = expit(np.array([-4.0, 3.0, 0.5]))
    assert np.allclose(w_b[1], ref_b / ref_b.sum() * 2.5, rtol=1e-14)   # unbiased values weight the output
    # ties: equal logits in one group go to the lower index
    lt = np.zeros((1, E), dtype=np.float32)
    x2, wg2 = _gate_case(lt)
    ids_t, _ = o.moe_gate(x2, wg2, np.zeros(E, dtype=np.float32), n_groups=G, topk_groups=2, top_k=3)
    assert ids_t[0].tolist() == [0, 1, 2]
    # random data: gate values sum to route_scale, ids distinct and inside kept groups
    rng = np.random.default_rng(25)
    xr = synth.normal_bf16(rng, (8, 256), 1.0)
    wr = synth.normal_bf16(rng, (64, 256), 0.05)
    br = rng.uniform(-0.1, 0.1, 64).astype(np.float32)
    ids_r, w_r = o.moe_gate(xr, wr, br)
    assert np.allclose(w_r.sum(axis=1), 2.5, rtol=1e-14)
    assert all(len(set(r)) == 8 for r in ids_r.tolist())
    assert all(len(set(e // 8 for e in r)) <= 4 for r in ids_r.tolist())


def pin_moe_route(o):
    """Routing tables against numpy's stable argsort of the selections by
    expert: offsets from the expert counts, tokens in order within an
    expert, rows_of_token the inverse map, gate values carried along."""
    rng = np.random.default_rng(26)
    T, k, E = 50, 4, 12
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[:, 0] = 3                                     # a busy expert; expert 11 may stay empty
    ids[ids == 11] = 10
    for t in range(T):                                # keep selections distinct per token
        if len(set(ids[t].tolist())) < k:
            ids[t] = [3, 0, 1, 2]
    w = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
    off, tor, rot, wor = o.moe_route(ids, w, E)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert np.array_equal(tor, (np.arange(T * k) // k)[order])
    assert np.array_equal(wor.view(np.uint32), w.reshape(-1)[order].view(np.uint32))
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(rot.reshape(-1), inv)
    assert off[11] == off[12]


def pin_act_quant_cols(o):
    """128x1 groups along the rows: bit for bit act_quant of the transpose
    (when M is a multiple of 128), a ragged last block equal to zero-padding
    it, and a power-of-two closed form (a column whose largest magnitude is
    448 * 2^a has scale 2^a and codes equal to x / 2^a)."""
    rng = np.random.default_rng(27)
    x = synth.activations(rng, 256, 384, n_outlier=3, outlier_scale=20.0)
    xq, sx = o.act_quant_cols(x)
    xqt, sxt = o.act_quant(np.ascontiguousarray(x.T))
    assert np.array_equal(xq, xqt.T)
    assert np.array_equal(sx.view(np.uint32), np.ascontiguousarray(sxt[:, :2].T).view(np.uint32))
    xr = synth.activations(rng, 200, 128)
    xqr, sxr = o.act_quant_cols(xr)
    pad = np.concatenate([xr, np.zeros((56, 128), dtype=np.uint16)])
    xqp, sxp = o.act_quant_cols(pad)
    assert np.array_equal(xqr, xqp[:200]) and np.array_equal(sxr.view(np.uint32), sxp.view(np.uint32))
    # closed form: column values are e4m3 codes times 2^-3, with 448 present
    v = e4m3_values()
    codes = _pos_codes_with_max(rng, 128)
    col = (v[codes] * 2.0 ** -3).astype(np.float32)
    xc = bf16_bits(np.stack([col, col * 0], axis=1))
    qc, sc = o.act_quant_cols(xc)
    assert sc[0, 0] == np.float32(2.0 ** -3) and np.array_equal(qc[:, 0], codes)
    assert sc[0, 1] == 0.0


def _exact_dgrad(dyq, sdy, wq, sw, m, k):
    vals = e4m3_values()
    tot = Fraction(0)
    for nb in range(dyq.shape[1] // 128):
        bsum = sum(Fraction(float(vals[dyq[m, n]])) * Fraction(float(vals[wq[n, k]]))
                   for n in range(nb * 128, (nb + 1) * 128))
        tot += Fraction(float(sdy[m, nb])) * Fraction(float(sw[nb, k // 128])) * bsum
    return tot


def pin_gemm_dgrad(o):
    """dX = dY W: bit for bit the forward GEMM with the weight and its block
    grid transposed (W^T is [K, N] with 128x128 blocks (kb, nb)), the
    dequantise-then-matmul form, and exact rationals on one element."""
    rng = np.random.default_rng(28)
    M, N, K = 40, 256, 384
    dy = synth.activations(rng, M, N, n_outlier=2, outlier_scale=10.0)
    w = synth.normal_bf16(rng, (N, K), 0.02)
    dyq, sdy = o.act_quant(dy)
    wq, sw = o.weight_quant(w)
    dx, L = o.gemm_dgrad(dyq, sdy, wq, sw)
    y_t, L_t = o.gemm(dyq, sdy, np.ascontiguousarray(wq.T), np.ascontiguousarray(sw.T))
    assert np.array_equal(dx, y_t) and np.array_equal(L, L_t)
    v = e4m3_values()
    dyd = v[dyq] * np.repeat(sdy[:, : N // 128].astype(np.float64), 128, 1)
    wd = v[wq] * np.repeat(np.repeat(sw.astype(np.float64), 128, 0), 128, 1)
    assert np.all(np.abs(dx - dyd @ wd) <= 1e-12 * L + 1e-300)
    m, k = 7, 300
    ex = _exact_dgrad(dyq, sdy, wq, sw, m, k)
    assert abs(Fraction(float(dx[m, k])) - ex) <= Fraction(2) ** -45 * Fraction(float(L[m, k]))


def pin_gemm_wgrad(o):
    """dW = dY^T X over the tokens with 128x1 groups: the dequantise-then-
    matmul form (numpy), exact rationals on one element, a ragged last block
    of tokens (200 = 128 + 72) that matters, and a rank-1 closed form: dY all
    1.75 = 448 * 2^-8 and X all 3.5 = 448 * 2^-7 (power-of-two scales, code
    448) give dW = 6.125 M exactly."""
    rng = np.random.default_rng(29)
    M, N, K = 200, 64, 96
    dy = synth.activations(rng, M, N, n_outlier=2, outlier_scale=10.0)
    x = synth.activations(rng, M, K)
    dyq, sdy = o.act_quant_cols(dy)
    xq, sx = o.act_quant_cols(x)
    dw, L = o.gemm_wgrad(dyq, sdy, xq, sx)
    v = e4m3_values()
    dyd = v[dyq] * np.repeat(sdy.astype(np.float64), 128, 0)[:M]
    xd = v[xq] * np.repeat(sx.astype(np.float64), 128, 0)[:M]
    assert np.all(np.abs(dw - dyd.T @ xd) <= 1e-12 * L + 1e-300)
    # the last 72 tokens contribute
    assert np.abs(dyd[128:].T @ xd[128:]).max() > 1e-3
    n, k = 5, 77
    ex = Fraction(0)
    for mb in range(2):
        bsum = sum(Fraction(float(v[dyq[m, n]])) * Fraction(float(v[xq[m, k]])) for m in range(mb * 128, min(M, mb * 128 + 128)))
        ex += Fraction(float(sdy[mb, n])) * Fraction(float(sx[mb, k])) * bsum
    assert abs(Fraction(float(dw[n, k])) - ex) <= Fraction(2) ** -45 * Fraction(float(L[n, k]))
    a = bf16_bits(np.full((M, 3), 1.75, dtype=np.float32))
    b = bf16_bits(np.full((M, 2), 3.5, dtype=np.float32))
    q1, s1 = o.act_quant_cols(a)
    q2, s2 = o.act_quant_cols(b)
    assert np.all(s1 == np.float32(2.0 ** -8)) and np.all(s2 == np.float32(2.0 ** -7))
    dw1, _ = o.gemm_wgrad(q1, s1, q2, s2)
    assert np.array_equal(dw1, np.full((3, 2), 6.125 * M))


def pin_act_quant_pow2(o):
    """Power-of-two scales: against exact rationals, s is a power of two with
    s/2 < amax/448 <= s; the codes are ml_dtypes' round-to-nearest-even e4m3
    of the exact quotient and never exceed 448; a group whose amax is
    448 * 2^a gets the same scale and codes as the fp32-scale path; all-zero
    groups get s = 0."""
    rng = np.random.default_rng(30)
    x = synth.activations(rng, 64, 512, n_outlier=5, outlier_scale=30.0)
    x[3, 128:256] = 0
    xq, sx = o.act_quant_pow2(x)
    xf = f32_of_bf16(x).astype(np.float64)
    v = e4m3_values()
    for m in range(64):
        for g in range(4):
            grp = xf[m, 128 * g:128 * (g + 1)]
            amax = np.abs(grp).max()
            s = float(sx[m, g])
            if amax == 0:
                assert s == 0.0 and not (xq[m, 128 * g:128 * (g + 1)] & 0x7F).any()
                continue
            mant, _ = np.frexp(s)
            assert mant == 0.5, "scale is not a power of two"
            ratio = Fraction(amax) / 448
            assert Fraction(s) / 2 < ratio <= Fraction(s)
            q = grp / s                                     # exact: power-of-two scaling
            assert np.abs(q).max() <= 448
            assert np.array_equal(xq[m, 128 * g:128 * (g + 1)], e4m3_code_lib(q))
            assert np.abs(v[xq[m, 128 * g:128 * (g + 1)]]).max() <= 448
    # amax = 448 * 2^a: the same as the fp32-scale path
    codes = _pos_codes_with_max(rng, 128)
    row = (v[codes] * 2.0 ** -5).astype(np.float32)
    xb = bf16_bits(row[None, :])
    q1, s1 = o.act_quant_pow2(xb)
    q2, s2 = o.act_quant(xb)
    assert s1[0, 0] == s2[0, 0] == np.float32(2.0 ** -5) and np.array_equal(q1, q2)


def pin_weight_quant_pow2(o):
    """Power-of-two weight scales per 128x128 block: against exact rationals
    (s a power of two with s/2 < amax/448 <= s over the block's valid rows),
    the codes ml_dtypes' round-to-nearest-even e4m3 of the exact quotient; a
    ragged last row block equals the zero-padded one; a block whose amax is
    448 * 2^a matches the fp32-scale path; an all-zero block has s = 0."""
    rng = np.random.default_rng(31)
    w = synth.normal_bf16(rng, (200, 384), 0.02)
    w[0:128, 128:256] = 0
    w[150, 300] = bf16_bits(np.array([[7.5]], dtype=np.float32))[0, 0]   # an outlier in the ragged block
    wq, sw = o.weight_quant_pow2(w)
    wf = f32_of_bf16(w).astype(np.float64)
    for nb in range(2):
        for kb in range(3):
            blk = wf[128 * nb:min(200, 128 * (nb + 1)), 128 * kb:128 * (kb + 1)]
            qb = wq[128 * nb:min(200, 128 * (nb + 1)), 128 * kb:128 * (kb + 1)]
            amax = np.abs(blk).max()
            s = float(sw[nb, kb])
            if amax == 0:
                assert s == 0.0 and not (qb & 0x7F).any()
                continue
            mant, _ = np.frexp(s)
            assert mant == 0.5, "scale is not a power of two"
            assert Fraction(s) / 2 < Fraction(amax) / 448 <= Fraction(s)
            assert np.array_equal(qb, e4m3_code_lib(blk / s))
    wp = np.zeros((256, 384), dtype=np.uint16)
    wp[:200] = w
    wq_p, sw_p = o.weight_quant_pow2(wp)
    assert np.array_equal(wq_p[:200], wq) and np.array_equal(sw_p.view(np.uint32), sw.view(np.uint32))
    v = e4m3_values()
    codes = np.stack([_pos_codes_with_max(rng, 128) for _ in range(128)])
    blk = bf16_bits((v[codes] * 2.0 ** -3).astype(np.float32))
    q1, s1 = o.weight_quant_pow2(blk)
    q2, s2 = o.weight_quant(blk)
    assert s1[0, 0] == s2[0, 0] == np.float32(2.0 ** -3) and np.array_equal(q1, q2)


ALL_PINS = [
    pin_codec_midpoints,
    pin_act_quant_rank1,
    pin_act_quant_division_exact,
    pin_act_quant_invariants,
    pin_weight_quant_blocks,
    pin_weight_quant_identity,
    pin_weight_quant_ragged,
    pin_weight_dequant,
    pin_gemm_bruteforce,
    pin_gemm_rank1,
    pin_gemm_diag,
    pin_gemm_vs_dequant_matmul,
    pin_grouped,
    pin_gemm_bias,
    pin_swiglu,
    pin_moe_dispatch,
    pin_moe_combine,
    pin_moe_gate,
    pin_moe_route,
    pin_act_quant_cols,
    pin_gemm_dgrad,
    pin_gemm_wgrad,
    pin_act_quant_pow2,
    pin_weight_quant_pow2,
]
