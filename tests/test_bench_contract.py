"""The JSON line bench.py prints, checked on the CPU where it can run there:
the reference arm (the oracle on the host cores) on the tiny workload, with
fp32 and with power-of-two scales, and
the committed DRAM-traffic table's lookup."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(not os.path.exists(os.path.join(ROOT, "oracle", "oracle.c")), reason="no oracle")
@pytest.mark.parametrize("workload", ["tiny", "tiny_pow2"])
def test_reference_arm_line(workload):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == workload
    if workload.endswith("_pow2"):
        assert "act_quant_pow2" in d["cpu_baseline"]["sample"]


def test_traffic_table_lookup():
    sys.path.insert(0, ROOT)
    import bench
    assert len(bench.kernel_sources_sha("fp8_gemm")) == 16
    # every committed capture is reported while its kernel's sources match it, else null
    with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as f:
        entries = [dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
                   for line in f if line.strip() and not line.startswith("#")]
    assert entries
    for kv in entries:
        t = bench.ncu_traffic(kv["kernel"], kv["workload"])
        assert (t is not None) == (kv["src_sha"] == bench.kernel_sources_sha(kv["kernel"]))
        if t is not None:
            assert t == float(kv["dram_bytes_per_launch"])
    assert bench.ncu_traffic("no_such_kernel", "kv_down") is None
