"""fp8bs_gemm_noalloc: the GEMM for callers that cannot allocate device memory
(allocator callbacks, plugin hosts that pass only inputs and outputs,
paths where a synchronising allocation is not allowed).  It takes its split-K
scratch from a fixed array inside the library instead of a caller workspace.

Called through the C ABI and compared, on two calls in a row, with the
existing entry point (fp8bs_gemm with a caller-allocated workspace) within the
GEMM bound the other tests use; the second call runs on scratch the first one
left behind.  This file is collected last so that a run stopping at the first
failure has run every other test first.
"""
import os
import re

import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import assert_gemm_close, bf16_to_f64, dev, host

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fp8bs.h")


def _scratch_limit() -> int:
    m = re.search(r"#define\s+FP8BS_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


def test_noalloc_gemm_matches_workspace_gemm_two_calls(orc):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs as F
    lib = F.lib
    limit = _scratch_limit()
    stream = torch.cuda.current_stream().cuda_stream
    for M in (128, 96):  # two calls in a row, different shapes (above the few-token kernel's 64)
        case = synth.q_down(M)
        xq_h, sx_h = orc.act_quant(case.x, lds=56)
        wq_h, sw_h = orc.weight_quant(case.w)
        xq, sx, wq, sw = dev(xq_h), dev(sx_h), dev(wq_h), dev(sw_h)
        N, K = wq_h.shape
        need = F.fp8bs_gemm_workspace_size(M, N, K)
        assert 0 < need <= limit, "this shape must take the split-K (scratch) plan"

        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        y_api = F.fp8bs_gemm(xq, sx, wq, sw, workspace=ws)

        y_new = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        st = lib.fp8bs_gemm_noalloc(xq.data_ptr(), sx.data_ptr(), sx.stride(0), wq.data_ptr(), sw.data_ptr(),
                                    M, N, K, y_new.data_ptr(), y_new.stride(0), stream)
        assert st == F.FP8BS_OK, F.fp8bs_status_string(st)
        assert F.fp8bs_sync_status() == F.FP8BS_OK

        y_ref, L = orc.gemm(xq_h, sx_h, wq_h, sw_h)
        # the same plan and the same in-order split-K reduction as the
        # existing entry point: identical bits
        assert torch.equal(y_new.view(torch.int16), y_api.view(torch.int16)), f"noalloc vs fp8bs_gemm M={M}"
        # and within the bound the GEMM tests use
        assert_gemm_close(host(y_new), bf16_to_f64(host(y_api)), L, f"noalloc vs fp8bs_gemm M={M}")
        # and both against the oracle
        assert_gemm_close(host(y_new), y_ref, L, f"noalloc vs oracle M={M}")
        assert_gemm_close(host(y_api), y_ref, L, f"fp8bs_gemm vs oracle M={M}")
