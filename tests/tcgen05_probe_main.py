"""Child-process body of test_gpu_tcgen05.py and of bench.py --probe-tcgen05:
runs the tcgen05 diagnostic entry point on seeded bf16 operands, compares each
result with a float64 host matmul of the same operands, and prints one JSON
line. Run as its own process so that a fault in it cannot poison the CUDA
context of the caller."""

from __future__ import annotations

import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from kimi_delta_attention_04_gb300 import _lib  # noqa: E402


def main() -> int:
    reps = int(sys.argv[1]) if len(sys.argv) > 1 else 200
    dev = torch.device("cuda", 0)
    gen = torch.Generator().manual_seed(7)
    checks, timings = [], []
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for layout in (0, 1):
        for a_tmem in (0, 1):
            for K in (16, 64, 128):
                for N in (16, 64, 256):
                    a = torch.randn(128, K, generator=gen).to(torch.bfloat16)
                    b = torch.randn(N, K, generator=gen).to(torch.bfloat16)
                    d, _ = _lib.selftest_tcgen05(a.to(dev), b.to(dev), layout=layout, a_from_tmem=a_tmem, err=err)
                    torch.cuda.synchronize()
                    ref = a.double() @ b.double().T
                    checks.append({"layout": layout, "a_from_tmem": a_tmem, "K": K, "N": N,
                                   "max_abs": float((d.cpu().double() - ref).abs().max()),
                                   "ref_max": float(ref.abs().max())})
    for K, N in ((16, 16), (16, 64), (16, 128), (16, 256), (128, 16), (128, 32), (128, 64), (128, 128)):
        a = torch.randn(128, K, generator=gen).to(torch.bfloat16).to(dev)
        b = torch.randn(N, K, generator=gen).to(torch.bfloat16).to(dev)
        for a_tmem in (0, 1):
            _, cyc = _lib.selftest_tcgen05(a, b, layout=1, a_from_tmem=a_tmem, reps=reps, err=err)
            torch.cuda.synchronize()
            c = cyc.cpu().tolist()
            n = max(c[3], 1)
            timings.append({"K": K, "N": N, "a_from_tmem": a_tmem, "mma_instructions": K // 16,
                            "issue_to_done_cycles": c[0] / n, "issue_to_data_cycles": c[1] / n,
                            "burst_cycles_per_group": c[2] / n, "reps": c[3],
                            "independent_accumulators": c[5],
                            "independent_burst_cycles_per_group": (c[4] / n) if c[5] else None,
                            "issue_cycles_per_group": c[6] / n})
    print(json.dumps({"err": int(err.item()), "checks": checks, "timings": timings}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
