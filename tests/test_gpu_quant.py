"""GPU parity of the quantisers and the dequantiser: bit-exact against the
oracle on the same seeded inputs, through the C ABI."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_bits_equal, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _act(F, orc, xbits, lds=None, ldx=None):
    M, K = xbits.shape
    kb = K // 128
    lds = lds or max(4, (kb + 3) // 4 * 4)
    if ldx is None:
        x = dev_bf16(xbits)
    else:  # strided input: rows ldx apart
        buf = np.zeros((M, ldx), np.uint16)
        buf[:, :K] = xbits
        x = dev_bf16(buf)[:, :K]
    sx = torch.full((M, lds), -7.0, dtype=torch.float32, device="cuda")
    xq, sx = F.fp8bs_act_quant(x, sx=sx)
    assert F.fp8bs_sync_status() == 0
    xq_ref, sx_ref = orc.act_quant(xbits, lds=lds)
    sx_h = host(sx)
    assert_bits_equal(host(xq), xq_ref, "xq")
    assert_bits_equal(sx_h[:, :kb], sx_ref[:, :kb], "sx")
    assert np.all(sx_h[:, kb:] == -7.0), "padding columns of sx must be untouched"


def test_act_quant_tiny(F, orc):
    _act(F, orc, synth.tiny().x)


@pytest.mark.parametrize("M", [1, 3, 16, 64, 129, 512])
def test_act_quant_q_shapes(F, orc, M):
    _act(F, orc, synth.q_down(M).x)


def test_act_quant_kv_full(F, orc):
    _act(F, orc, synth.kv_down().x)


def test_act_quant_large_full(F, orc):
    _act(F, orc, synth.large_square().x)


def test_act_quant_strided_and_padded(F, orc):
    x = synth.activations(np.random.default_rng(5), 37, 640)
    _act(F, orc, x, lds=12, ldx=648)


def test_act_quant_special_groups(F, orc):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 1024)).astype(np.float32)
    x[0, :128] = 0.0
    x[0, 128:256] = -0.0
    x[1, :128] = 1e-38                         # fp32-subnormal-range bf16 values
    x[1, 128:256] = rng.standard_normal(128).astype(np.float32) * np.float32(1e-30)
    x[2, :128] = 3e38                          # near the bf16 maximum
    x[3, :128] = 0.0
    x[3, 7] = -2.5                             # single nonzero
    x[4, :] = 448.0
    x[5, 256:384] = np.linspace(-1, 1, 128)
    xb = synth.to_bf16_bits(x)
    xb[6, :128] = np.arange(128, dtype=np.uint16)            # bf16 subnormals / tiny patterns
    xb[7, :128] = 0x8000 | np.arange(128, dtype=np.uint16)
    _act(F, orc, xb)


def test_act_quant_division_sweep(F, orc):
    """Every positive bf16 value below amax, for many amax: the quotient x/s
    lands on every part of the e4m3 grid, including rounding boundaries."""
    rng = np.random.default_rng(7)
    xs = np.arange(0x0001, 0x7F80, dtype=np.uint16)          # all finite positive bf16
    amaxes = rng.integers(0x3800, 0x4700, size=48).astype(np.uint16)
    rows = []
    for a in amaxes:
        cand = xs[xs < a]
        cand = cand[rng.permutation(cand.size)][: 127 * 64]
        n = cand.size // 127 * 127
        g = np.empty((n // 127, 128), np.uint16)
        g[:, 0] = a
        g[:, 1:] = cand[:n].reshape(-1, 127)
        g[1::2, 1::3] |= 0x8000                                  # mixed signs
        rows.append(g.reshape(-1))
    flat = np.concatenate(rows)
    flat = flat[: flat.size // 1024 * 1024]
    _act(F, orc, flat.reshape(-1, 1024))


def _wq(F, orc, wbits):
    w = dev_bf16(wbits)
    wq, sw = F.fp8bs_weight_quant(w)
    assert F.fp8bs_sync_status() == 0
    wq_ref, sw_ref = orc.weight_quant(wbits)
    assert_bits_equal(host(wq), wq_ref, "wq")
    assert_bits_equal(host(sw), sw_ref, "sw")
    wd = F.fp8bs_weight_dequant(wq, sw)
    assert F.fp8bs_sync_status() == 0
    assert_bits_equal(host(wd), orc.weight_dequant(wq_ref, sw_ref), "dequant")


def test_weight_quant_tiny(F, orc):
    _wq(F, orc, synth.tiny().w)


def test_weight_quant_kv_ragged(F, orc):
    _wq(F, orc, synth.kv_down(M=1).w)


def test_weight_quant_q(F, orc):
    _wq(F, orc, synth.q_down(1).w)


def test_weight_quant_large_full(F, orc):
    _wq(F, orc, synth.large_square(M=1).w)


@pytest.mark.parametrize("N", [1, 5, 127, 130, 200])
def test_weight_quant_ragged_rows(F, orc, N):
    rng = np.random.default_rng(N)
    w = synth.normal_bf16(rng, (N, 384), 0.05)
    w[0, :5] = 0
    _wq(F, orc, w)


def test_weight_quant_identity_and_zero_blocks(F, orc):
    _wq(F, orc, synth.to_bf16_bits(np.eye(512, dtype=np.float32)))


def test_weight_dequant_all_codes(F, orc):
    """Every non-NaN code under several scales (incl. 0 and tiny ones)."""
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 256, size=(256, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E
    codes[0, :256] = np.arange(256)
    codes[0, [0x7F, 0xFF]] = 0
    sw = np.array([[1.0, 0.0, 3.1e-5, 7.77], [1e-30, 2.0 ** -20, 123.5, 0.1]], np.float32)
    wd = F.fp8bs_weight_dequant(dev(codes), dev(sw))
    assert F.fp8bs_sync_status() == 0
    assert_bits_equal(host(wd), orc.weight_dequant(codes, sw), "dequant")


def test_e4m3_encoder_exhaustive(F, orc):
    """All 2^32 fp32 bit patterns through the device encoder against the
    oracle's encoder (NaN inputs: any NaN code accepted)."""
    chunk = 1 << 26
    for c in range((1 << 32) // chunk):
        bits = np.arange(c * chunk, (c + 1) * chunk, dtype=np.uint64).astype(np.uint32)
        v = bits.view(np.float32)
        got = host(F.fp8bs_e4m3_encode_f32(dev(v)))
        want = orc.e4m3_encode(v)
        nan_in = (bits & 0x7FFFFFFF) > 0x7F800000
        ok = (got == want) | (nan_in & ((got & 0x7F) == 0x7F))
        bad = np.nonzero(~ok)[0]
        assert bad.size == 0, [(hex(int(bits[i])), hex(got[i]), hex(want[i])) for i in bad[:5]]


def _every_pair_batches(elems_per_batch=1 << 27):
    """Groups [amax, x_1 .. x_127] covering, for every positive finite bf16
    amax, every bf16 x (both signs) with |x| <= amax; yielded in batches of
    rows of 1024 elements (8 groups)."""
    codes = np.arange(0x0001, 0x7F80, dtype=np.uint32)   # positive finite bf16, increasing value
    pending, size = [], 0
    for c in codes:
        mags = np.arange(0, c + 1, dtype=np.uint32)
        xs = np.concatenate([mags, mags | 0x8000]).astype(np.uint16)
        n_groups = -(-xs.size // 127)
        g = np.zeros((n_groups, 128), np.uint16)
        g[:, 0] = c
        g[:, 1:].reshape(-1)[: xs.size] = xs
        pending.append(g)
        size += g.size
        if size >= elems_per_batch:
            yield _rows_of_1024(pending)
            pending, size = [], 0
    if pending:
        yield _rows_of_1024(pending)


def _rows_of_1024(groups):
    flat = np.concatenate(groups).reshape(-1)
    pad = (-flat.size) % 1024
    if pad:
        flat = np.concatenate([flat, np.zeros(pad, np.uint16)])
    return flat.reshape(-1, 1024)


def test_act_quant_every_amax_x_pair(F, orc):
    """Exhaustive over the quantisers' arithmetic domain: for every positive
    finite bf16 amax and every bf16 x with |x| <= amax (about 1.07e9 pairs),
    the device codes and scales equal the oracle's RN32(x / (amax/448))
    encoding bit for bit.  The group's other members do not enter x's code,
    so this covers every input of act_quant and weight_quant."""
    total = 0
    for xb in _every_pair_batches():
        x = dev_bf16(xb)
        xq, sx = F.fp8bs_act_quant(x)
        assert F.fp8bs_sync_status() == 0
        xq_ref, sx_ref = orc.act_quant(xb, lds=sx.shape[1])
        assert_bits_equal(host(xq), xq_ref, "xq")
        assert_bits_equal(host(sx)[:, :8], sx_ref[:, :8], "sx")
        total += xb.size
        del x, xq, sx
    assert total > 1_000_000_000
