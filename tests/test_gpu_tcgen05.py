"""The tcgen05 diagnostic (kda_selftest_tcgen05) through the C ABI: one
5th-generation tensor-core MMA per case, with the operands in shared memory
(no swizzle and 128-byte swizzle) or A in tensor memory, checked element by
element against a float64 host matmul of the same bf16 operands, and the timed
round trips reported. Runs in a child process (tcgen05_probe_main.py)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    from kimi_delta_attention_04_gb300 import build
    build.build()
    out = subprocess.run([sys.executable, os.path.join(HERE, "tcgen05_probe_main.py"), "100"], capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_tcgen05_mma_matches_host_matmul(probe):
    assert probe["err"] == 0
    assert len(probe["checks"]) == 36
    for c in probe["checks"]:
        # fp32 accumulation of K <= 128 bf16 products of N(0,1) values
        assert c["max_abs"] <= 1e-3 * max(1.0, c["ref_max"]), c


def test_tcgen05_round_trip_is_measured(probe):
    for t in probe["timings"]:
        assert t["reps"] == 100
        assert 0 < t["issue_to_done_cycles"] <= t["issue_to_data_cycles"] < 1e6, t
        assert t["burst_cycles_per_group"] > 0, t
    print(json.dumps(probe["timings"], indent=1))
