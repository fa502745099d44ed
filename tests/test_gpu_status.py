"""The failure path on the GPU without a fault: a bounded wait that nothing
completes expires, the kernel records it and returns, the host reads
FP8BS_ERR_TIMEOUT, and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def test_wait_timeout_is_reported_and_cleared(F):
    assert F.fp8bs_sync_status() == F.FP8BS_OK
    F.fp8bs_debug_wait_timeout(2_000_000)  # 2 ms
    assert F.fp8bs_sync_status() == F.FP8BS_ERR_TIMEOUT
    assert F.fp8bs_sync_status() == F.FP8BS_OK  # cleared by the read
    # the context still works
    x = torch.randn(4, 128, device="cuda").to(torch.bfloat16)
    xq, sx = F.fp8bs_act_quant(x)
    assert F.fp8bs_sync_status() == F.FP8BS_OK


def test_argument_errors_raise(F):
    x = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(F.Fp8bsError) as e:
        F.fp8bs_act_quant(x)
    assert e.value.status == F.FP8BS_ERR_UNSUPPORTED
    x = torch.zeros(4, 136, dtype=torch.bfloat16, device="cuda")[:, 1:129]
    with pytest.raises(F.Fp8bsError) as e:
        F.fp8bs_act_quant(x)
    assert e.value.status == F.FP8BS_ERR_MISALIGNED


def test_library_is_the_in_tree_build(F):
    import os
    assert os.path.abspath(F.LIB_PATH).startswith(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    maps = open("/proc/self/maps").read()
    assert "libfp8bs.so" in maps
