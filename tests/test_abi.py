"""Host-only checks of the C-ABI library: it loads, exports every declared
symbol, and rejects bad arguments before touching any device."""
import ctypes

import pytest

fp8bs = pytest.importorskip("fp8_block_scaled_18_b300.fp8bs")
lib = fp8bs.lib

A = 0x10000  # a 16-byte-aligned fake address; validation fails before any use


def test_exports_every_declared_symbol():
    names = fp8bs.declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    for required in ("fp8bs_act_quant", "fp8bs_weight_quant", "fp8bs_weight_dequant", "fp8bs_gemm",
                     "fp8bs_grouped_gemm", "fp8bs_sync_status", "fp8bs_status_string"):
        assert required in names


def test_binding_covers_the_header():
    """Every call the header declares has a typed ctypes signature and a
    Python function of the same name, and the binding declares nothing the
    header does not."""
    declared = set(fp8bs.declared_symbols())
    assert declared == set(fp8bs._SIGS)
    for n in declared:
        assert callable(getattr(fp8bs, n)), n


def test_status_strings_and_version():
    for s in range(7):
        assert fp8bs.fp8bs_status_string(s).startswith("FP8BS")
    assert fp8bs.fp8bs_status_string(99) == "FP8BS: unknown status"
    assert fp8bs.fp8bs_version() == (0 << 16) | (1 << 8)


def test_act_quant_validation():
    f = lib.fp8bs_act_quant
    assert f(A, -1, 128, 128, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, 4, 100, 128, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert f(A, 4, 0, 128, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert f(A, 0, 128, 128, A, 128, A, 4, None) == fp8bs.FP8BS_OK          # empty: no-op
    assert f(None, 4, 128, 128, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, 4, 256, 128, A, 256, A, 4, None) == fp8bs.FP8BS_ERR_INVALID_ARG  # ldx < K
    assert f(A, 4, 256, 256, A, 256, A, 1, None) == fp8bs.FP8BS_ERR_INVALID_ARG  # lds < K/128
    assert f(A + 2, 4, 128, 128, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert f(A, 4, 128, 132, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_MISALIGNED   # ldx % 8
    assert f(A, 4, 128, 128, A, 136, A, 4, None) == fp8bs.FP8BS_ERR_MISALIGNED   # ldq % 16
    assert f(A, 4, 128, 128, A, 128, A, 6, None) == fp8bs.FP8BS_ERR_MISALIGNED   # lds % 4


def test_weight_calls_validation():
    assert lib.fp8bs_weight_quant(A, 10, 129, A, A, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert lib.fp8bs_weight_quant(A, -5, 128, A, A, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert lib.fp8bs_weight_quant(A, 0, 128, A, A, None) == fp8bs.FP8BS_OK
    assert lib.fp8bs_weight_quant(A + 8, 10, 128, A, A, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert lib.fp8bs_weight_quant(A, 128 * 65536, 128, A, A, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert lib.fp8bs_weight_dequant(A, A, 10, 64, A, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert lib.fp8bs_weight_dequant(A, None, 10, 128, A, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert lib.fp8bs_weight_dequant(A, A, 10, 128, A + 4, None) == fp8bs.FP8BS_ERR_MISALIGNED


def test_gemm_validation():
    g = lib.fp8bs_gemm
    assert g(A, A, 4, A, A, 4, 8, 200, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert g(A, A, 4, A, A, -4, 8, 128, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert g(A, A, 4, A, A, 0, 8, 128, A, 8, None, 0, None) == fp8bs.FP8BS_OK
    assert g(A, A, 4, A, A, 4, 0, 128, A, 8, None, 0, None) == fp8bs.FP8BS_OK
    assert g(A, A, 4, None, A, 4, 8, 128, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert g(A, A, 4, A, A, 4, 16, 128, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_INVALID_ARG  # ldy < N
    assert g(A, A, 4, A, A, 4, 8, 128, A, 12, None, 0, None) == fp8bs.FP8BS_ERR_MISALIGNED  # ldy % 8
    assert g(A, A, 2, A, A, 4, 8, 128, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_MISALIGNED   # lds % 4
    assert g(A + 1, A, 4, A, A, 4, 8, 128, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert g(A, A, 4, A, A, 4, 8, 128, A, 8, A + 4, 64, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert g(A, A, 4, A, A, 1 << 31, 8, 128, A, 8, None, 0, None) == fp8bs.FP8BS_ERR_UNSUPPORTED


def test_gemm_fused_validation():
    f = lib.fp8bs_gemm_fused
    ok = fp8bs.FP8BS_OK
    # (xq, sx, lds, wq, sw, bias, M, N, K, y, ldy, yq, ldyq, sy, ldsy, stream)
    assert f(A, A, 4, A, A, None, 0, 256, 128, A, 256, None, 0, None, 0, None) == ok  # M == 0: no-op
    assert f(A, A, 4, A, A, None, 4, 256, 128, None, 0, None, 0, None, 0, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, A, 4, A, A, None, 4, 256, 100, A, 256, None, 0, None, 0, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    # yq needs whole 128-column groups, an sy, and 16-byte rows
    assert f(A, A, 4, A, A, None, 4, 200, 128, None, 0, A, 208, A, 4, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert f(A, A, 4, A, A, None, 4, 256, 128, None, 0, A, 256, None, 4, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, A, 4, A, A, None, 4, 256, 128, None, 0, A, 200, A, 4, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, A, 4, A, A, None, 4, 256, 128, None, 0, A, 264, A, 4, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert f(A, A, 4, A, A, None, 4, 256, 128, None, 0, A, 256, A, 1, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, A, 4, A, A, None, 4, 256, 128, None, 0, A, 256, A + 4, 4, None) == fp8bs.FP8BS_ERR_MISALIGNED
    # y rules as fp8bs_gemm; the bias needs 2-byte alignment only
    assert f(A, A, 4, A, A, None, 4, 256, 128, A, 260, None, 0, None, 0, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert f(A, A, 4, A, A, A + 1, 4, 256, 128, A, 256, None, 0, None, 0, None) == fp8bs.FP8BS_ERR_MISALIGNED


def test_grouped_swiglu_validation():
    f = lib.fp8bs_grouped_gemm_swiglu
    # (xq, sx, lds, w1q, sw1, w3q, sw3, off, G, T, I, K, h, ldh, hq, ldhq, sh, ldsh, stream)
    args = [A, A, 4, A, A, A, A, A, 4, 64, 256, 128, A, 256, None, 0, None, 0, None]
    assert f(*args[:9], 0, *args[10:]) == fp8bs.FP8BS_OK                         # no rows: no-op
    bad = list(args); bad[10] = 200
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # I % 128
    bad = list(args); bad[5] = None
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # no w3
    bad = list(args); bad[12] = None
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # neither h nor hq
    bad = list(args); bad[14], bad[15], bad[16], bad[17] = A, 256, None, 4
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # hq without sh
    bad = list(args); bad[14], bad[15], bad[16], bad[17] = A, 264, A, 4
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # ldhq % 16
    bad = list(args); bad[6] = A + 2
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # sw3 alignment


def test_gemm_noalloc_validation():
    """The no-allocation GEMM rejects bad arguments before any CUDA call."""
    f = lib.fp8bs_gemm_noalloc
    assert f(A, A, 4, A, A, 4, 8, 200, A, 8, None) == fp8bs.FP8BS_ERR_UNSUPPORTED   # K % 128
    assert f(A, A, 4, A, A, -1, 8, 128, A, 8, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert f(A, A, 4, A, A, 0, 8, 128, A, 8, None) == fp8bs.FP8BS_OK                # empty: a no-op
    assert f(A, A, 4, None, A, 4, 8, 128, A, 8, None) == fp8bs.FP8BS_ERR_INVALID_ARG


def test_backward_calls_validation():
    """The column quantiser and the weight-gradient GEMM reject bad arguments
    before any CUDA call."""
    q = lib.fp8bs_act_quant_cols
    assert q(A, 4, 100, 128, A, 16, A, 128, None) == fp8bs.FP8BS_ERR_UNSUPPORTED     # K % 64
    assert q(A, -1, 64, 64, A, 16, A, 64, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert q(A, 0, 64, 64, A, 16, A, 64, None) == fp8bs.FP8BS_OK                     # empty: a no-op
    assert q(A, 40, 64, 64, A, 32, A, 64, None) == fp8bs.FP8BS_ERR_INVALID_ARG       # ldt < M
    assert q(A, 40, 64, 64, A, 40, A, 64, None) == fp8bs.FP8BS_ERR_MISALIGNED        # ldt % 16
    assert q(A, 40, 64, 60, A, 48, A, 64, None) == fp8bs.FP8BS_ERR_INVALID_ARG       # ldx < K
    g = lib.fp8bs_gemm_wgrad
    ok = [A, 32, A, 64, A, 32, A, 128, 32, 64, 128, A, 128, None]
    bad = list(ok); bad[8] = 0
    assert g(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                      # T == 0
    bad = list(ok); bad[9] = 0
    assert g(*bad) == fp8bs.FP8BS_OK                                                   # N == 0: a no-op
    bad = list(ok); bad[1] = 24
    assert g(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                      # lddyt < T
    bad = list(ok); bad[1] = 40
    assert g(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                       # lddyt % 16
    bad = list(ok); bad[7] = 130
    assert g(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                       # ldsx % 4
    bad = list(ok); bad[11] = A + 4
    assert g(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                       # dw alignment
    bad = list(ok); bad[2] = None
    assert g(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG


def test_grouped_validation():
    gg = lib.fp8bs_grouped_gemm
    assert gg(A, A, 4, A, A, None, 4, 16, 8, 128, A, 8, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert gg(A, A, 4, A, A, A, -1, 16, 8, 128, A, 8, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert gg(A, A, 4, A, A, A, 4, 0, 8, 128, A, 8, None) == fp8bs.FP8BS_OK
    assert gg(A, A, 4, A, A, A, 2000, 16, 8, 128, A, 8, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    assert gg(A, A, 4, A, A, A + 2, 4, 16, 8, 128, A, 8, None) == fp8bs.FP8BS_ERR_MISALIGNED
    assert gg(A, A, 4, A, A, A, 4, 16, 8, 136, A, 8, None) == fp8bs.FP8BS_ERR_UNSUPPORTED
    # the tile table lives in shared memory: no scratch for any shape
    assert lib.fp8bs_grouped_gemm_workspace_size(256, 2048, 7168) == 0


def test_moe_dispatch_validation():
    f = lib.fp8bs_moe_dispatch
    # (xq, ldq, sx, lds, tokens, K, token_of_row, R, xq_rows, ldq_rows, sx_rows, lds_rows, stream)
    args = [A, 256, A, 4, 16, 256, A, 32, A, 256, A, 4, None]
    ok = fp8bs.FP8BS_OK
    assert f(*args[:7], 0, *args[8:]) == ok                                       # no rows: no-op
    bad = list(args); bad[5] = 200
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # K % 128
    bad = list(args); bad[4] = 0
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # rows but no tokens
    bad = list(args); bad[6] = None
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # no map
    bad = list(args); bad[9] = 128
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # ldq_rows < K
    bad = list(args); bad[11] = 1
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # lds_rows < K/128
    bad = list(args); bad[1] = 264
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # ldq % 16
    bad = list(args); bad[8] = A + 8
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # xq_rows alignment
    bad = list(args); bad[6] = A + 2
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # map alignment
    bad = list(args); bad[7] = -1
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG


def test_moe_combine_validation():
    f = lib.fp8bs_moe_combine
    # (yk, ldyk, R, w, rows_of_token, tokens, topk, dim, z, ldz, y, ldy, stream)
    Y = A + 0x100000  # y far from z
    args = [A, 128, 64, A, A, 8, 8, 128, None, 0, Y, 128, None]
    ok = fp8bs.FP8BS_OK
    assert f(*args[:5], 0, *args[6:]) == ok                                       # no tokens: no-op
    bad = list(args); bad[7] = 100
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # dim % 8
    bad = list(args); bad[2] = 0
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # routed but no rows
    bad = list(args); bad[10] = None
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # no y
    bad = list(args); bad[1] = 64
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # ldyk < dim
    bad = list(args); bad[1] = 132
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # ldyk % 8
    bad = list(args); bad[3] = A + 2
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # w alignment
    bad = list(args); bad[8], bad[9] = Y + 256, 128
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # z overlaps y
    bad = list(args); bad[8], bad[9] = A + 0x200008, 128
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # z alignment
    bad = list(args); bad[6] = -1
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG


def test_moe_gate_validation():
    f = lib.fp8bs_moe_gate
    # (x, ldx, wg, bias, T, dim, E, n_groups, topk_groups, top_k, route_scale, ids, weights, stream)
    args = [A, 7168, A, A, 64, 7168, 256, 8, 4, 8, 2.5, A, A, None]
    assert f(*args[:4], 0, *args[5:]) == fp8bs.FP8BS_OK                          # no tokens: no-op
    bad = list(args); bad[5] = 7000
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # dim % 64
    bad = list(args); bad[6] = 264
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # E > 256
    bad = list(args); bad[7] = 7
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # groups do not divide E
    bad = list(args); bad[8] = 9
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # keep more groups than exist
    bad = list(args); bad[9] = 17
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # top_k > 16
    bad = list(args); bad[7], bad[8], bad[9] = 32, 1, 9
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG                                 # top_k > experts kept
    bad = list(args); bad[1] = 7172
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # ldx % 8
    bad = list(args); bad[2] = A + 8
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED                                  # wg alignment
    bad = list(args); bad[11] = None
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG


def test_moe_route_validation():
    f = lib.fp8bs_moe_route
    # (ids, weights, T, top_k, E, offsets, token_of_row, rows_of_token, weight_of_row, stream)
    args = [A, A, 64, 8, 256, A, A, A, A, None]
    bad = list(args); bad[4] = 300
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # E > 256
    bad = list(args); bad[3] = 17
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # top_k > 16
    bad = list(args); bad[3] = 0
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG
    bad = list(args); bad[6] = None
    assert f(*bad) == fp8bs.FP8BS_ERR_INVALID_ARG
    bad = list(args); bad[7] = A + 2
    assert f(*bad) == fp8bs.FP8BS_ERR_MISALIGNED
    bad = list(args); bad[2] = 2 ** 29
    assert f(*bad) == fp8bs.FP8BS_ERR_UNSUPPORTED                                 # more routed rows than int32


def test_debug_calls_validation():
    assert lib.fp8bs_debug_wait_timeout(0, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert lib.fp8bs_e4m3_encode_f32(A, -1, A, None) == fp8bs.FP8BS_ERR_INVALID_ARG
    assert lib.fp8bs_e4m3_encode_f32(A, 0, A, None) == fp8bs.FP8BS_OK


def test_valid_call_without_a_device_fails_loudly():
    """On a machine with no GPU a well-formed call reports FP8BS_ERR_CUDA:
    there is no CPU path to fall back to."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.fp8bs_act_quant(A, 4, 128, 128, A, 128, A, 4, None) == fp8bs.FP8BS_ERR_CUDA
    assert lib.fp8bs_gemm_workspace_size(1, 1536, 7168) == 0
    # in-place combine (z is y) passes validation and then needs the device
    assert lib.fp8bs_moe_combine(A, 128, 64, A, A, 8, 8, 128, A + 0x100000, 128, A + 0x100000, 128,
                                 None) == fp8bs.FP8BS_ERR_CUDA
