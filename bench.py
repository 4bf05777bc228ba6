"""Benchmark of the KDA hot path on GB300.

One step = one chunk forward over the prefill workload (bf16, B=1, H=32,
T=8192, d=128, gate inputs, beta logits, L2 norm, fp32 h0) followed by one fused
decode step over the decode workload (B=256, H=HV=32, K=V=128, fp32 slot pool
[512, 32, 128, 128], 26 padding rows). Inputs are seeded synthetic data,
resident in HBM before timing; every input is larger than L2, so no flush is
needed between steps.

Prints ONE JSON line (rank 0). value = chunk-forward tokens/s (whole job), with
decode microseconds per step, both roofline fractions, the e2e figure through
host buffers, the oracle's CPU throughput and the clocks seen while timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle as it stands (the reference arm
of this benchmark): whole steps of the same workload (the full prefill forward,
then the full decode step), spread over every host core by a process pool
(prefill by heads, decode by rows). cpu_baseline in the GPU arm's line is the
same oracle on the same cores. Under torchrun each rank runs its own replica
of the workload (weak scaling; the path needs no collective).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "KDA chunk-fwd tokens/s (H=32,d=128) + % roofline; decode μs/step at B=256"
UNIT = "tokens/s"
WORKLOAD = "KDA prefill bf16 B=1 H=32 T=8192 dk=dv=128 (gate inputs, beta logits, L2 norm, h0) + fused decode B=256 H=HV=32 K=V=128 (fp32 pool 512 slots, 26 pads)"

# Algorithmic bytes (each input read once, each output written once).
PREFILL_T, PREFILL_H, D = 8192, 32, 128
BYTES_PER_TOKEN = PREFILL_H * (D * 2 * 3 + D * 4 + 2 + D * 2)  # q,k,v bf16 + a fp32 + b bf16 + o bf16 = 49,216
STATE_BYTES = PREFILL_H * D * D * 4                            # one fp32 state set (h0 or hT)
PARAM_BYTES = PREFILL_H * D * 4 + PREFILL_H * 4                # dt_bias + A_log


def prefill_algorithmic_bytes(T=PREFILL_T):
    return T * BYTES_PER_TOKEN + 2 * STATE_BYTES + PARAM_BYTES


def prefill_algorithmic_flops(T=PREFILL_T):
    """Tensor work per token and head of the chunk form (C = 16, d = 128):
    K_dec S, Q_dec S (2 * 2 d^2), state update K_res^T U (2 d^2), L and Mqk
    (2 * 2 * C d / 2, lower triangles), Mqk U (C d), INV (Neumann, 6 C^2 per token),
    W and U~ (2 * 2 C d)."""
    C = 16
    per = 4 * D * D + 2 * D * D + 2 * C * D + C * D + 6 * C * C + 4 * C * D
    return T * PREFILL_H * per


def recurrent_algorithmic_bytes(n_valid, B, T, H=32, HV=32, K=128, V=128):
    """Short-T recurrent step: each valid row's slot read and written once for
    its T tokens, the valid rows' q, k, v, a, b, every row's o, the parameters."""
    state = n_valid * HV * V * K * 4 * 2
    io = n_valid * T * (2 * H * K * 2 + HV * V * 2 + HV * K * 2 + HV * 2)
    params = HV * 4 + HV * K * 4 + B * 4
    return state + io + params + B * T * HV * V * 2


def decode_algorithmic_bytes(n_valid, H=32, HV=32, K=128, V=128, B=256):
    state = n_valid * HV * V * K * 4 * 2                            # read + write of each valid slot
    io = n_valid * (2 * H * K * 2 + HV * V * 2 + HV * K * 2 + HV * 2)  # packed q,k,v + a + b of valid rows
    params = HV * 4 + HV * K * 4 + B * 4                               # A_log, dt_bias, indices
    return state + io + params + B * HV * V * 2                         # + o


# Sources of the kernels the roofline objects describe (a stored ncu traffic
# figure is only reported while these files are unchanged).
CHUNK_KERNEL_SOURCES = ["kda_chunk_fused.cu", "kda_common.cuh", "kda_cluster.cuh", "kda_tma.h", "kda_tma.cpp"]
DECODE_KERNEL_SOURCES = ["kda_decode.cu", "kda_common.cuh"]
RECURRENT_KERNEL_SOURCES = ["kda_recurrent_tc.cu", "kda_common.cuh", "kda_cluster.cuh", "kda_tcgen05.cuh"]
RECURRENT_B, RECURRENT_T, RECURRENT_SLOTS = 128, 8, 256  # speculative-style step: 128 rows x 8 tokens
RECURRENT_LONG_B, RECURRENT_LONG_T = 64, 64              # the longest T the entry point takes
CHUNK_LAUNCHES_PER_STEP = 1   # kda_chunk_fused_kernel (bf16, d = 128, no cu_seqlens)
DECODE_LAUNCHES_PER_STEP = 1  # kda_decode_kernel


# GB300's nominal HBM3e bandwidth (8 stacks, 7.9 TB/s): a second denominator for the
# roofline fractions, beside the measured copy bandwidth they are quoted against.
SPEC_HBM_GBS = 7900.0


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_sources_sha(names):
    h = hashlib.sha256()
    for n in names:
        h.update((ROOT / "kimi_delta_attention_04_gb300" / "csrc" / n).read_bytes())
    return h.hexdigest()[:16]


def stored_traffic(kernel_key, sha, units=1.0):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    profiles/traffic.txt, if it was taken on the current kernel source, scaled
    by `units` (the ratio of this launch's work to the captured launch's);
    otherwise None. Lines: <kernel> source_sha=<sha> dram_bytes=<n> units=<u> ..."""
    p = ROOT / "profiles" / "traffic.txt"
    if not p.exists():
        return None
    for line in p.read_text().splitlines():
        parts = line.split()
        if not parts or parts[0] != kernel_key:
            continue
        kv = dict(x.split("=", 1) for x in parts[1:] if "=" in x)
        if kv.get("source_sha") != sha:
            return None
        return float(kv["dram_bytes"]) * units / float(kv.get("units", "1"))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device):
    """The element-wise maximum of `values` (floats) over the ranks of the
    default process group (NCCL on GPUs, gloo on CPU); the values themselves
    with one rank. Every rank gets the result."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def bench_config(world):
    """The `config` object of the benchmark line, the same for both arms."""
    return {"workload": WORKLOAD, "global_batch": world, "seq_len": PREFILL_T,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (prefill 403 MB, decode ~964 MB touched); no flush",
            "step": "one chunk forward (prefill) then one decode step (B=256)"}


# --- the fp64 oracle on the host cores: a process pool over heads (prefill) and
# rows (decode). Workers are started with `spawn` (safe after CUDA is in use)
# and run numpy/torch single-threaded, one worker per core. ---

def _pool_init():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    sys.path.insert(0, str(ROOT))
    import torch
    torch.set_num_threads(1)


_SHM = {}  # worker side: shared arrays attached once, by name


def _shared(spec):
    """Worker: numpy view of a shared-memory array (name, shape, dtype)."""
    import numpy as np
    from multiprocessing import shared_memory
    name, shape, dtype = spec
    if name not in _SHM:
        shm = shared_memory.SharedMemory(name=name)
        _SHM[name] = (shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf))
    return _SHM[name][1]


def _oracle_prefill_part(task):
    """Worker: the token-recurrence oracle on some heads of the prefill; seconds."""
    from oracle import kda_oracle as ko
    specs, heads, scale = task
    q, k, v, a, dt_bias, A_log, b, h0 = (_shared(x) for x in specs)
    T, H, K = q.shape[1], q.shape[2], q.shape[3]
    t0 = time.perf_counter()
    ko.kda_forward(q[:, :, heads], k[:, :, heads], v[:, :, heads], scale=scale,
                   a=a.reshape(1, T, H, K)[:, :, heads].reshape(1, T, -1),
                   dt_bias=dt_bias.reshape(H, K)[heads].reshape(-1), A_log=A_log[heads], b=b[:, :, heads],
                   h0=h0[:, heads], l2norm_qk=True)
    return time.perf_counter() - t0


def _oracle_decode_part(task):
    """Worker: the decode oracle on some rows (their slots compacted); seconds."""
    from oracle import kda_oracle as ko
    specs, rows, local, dims = task
    packed, a, b, A_log, dt_bias, pool, idx = (_shared(x) for x in specs)
    slots = idx[rows]
    sub = pool[slots[slots >= 0]]
    t0 = time.perf_counter()
    ko.kda_decode(packed[rows], a[rows], b[rows], A_log, dt_bias, sub, local, **dims)
    return time.perf_counter() - t0


class OracleCpu:
    """The oracle spread over `cores` worker processes: prefill by heads, decode
    by rows. Inputs are the benchmark's own seeded workloads (first T tokens),
    placed once in shared memory, so a timed map only sends indices."""

    def __init__(self, T=PREFILL_T, cores=None, with_decode=True):
        import multiprocessing as mp

        import numpy as np
        from multiprocessing import shared_memory

        from kimi_delta_attention_04_gb300 import workloads as W
        self.cores = int(cores or os.cpu_count() or 1)
        self.T = T
        self._shm = []

        def put(t):
            x = np.ascontiguousarray(t.float().numpy() if t.dtype != __import__("torch").int32 else t.numpy())
            shm = shared_memory.SharedMemory(create=True, size=max(x.nbytes, 1))
            np.ndarray(x.shape, dtype=x.dtype, buffer=shm.buf)[...] = x
            self._shm.append(shm)
            return (shm.name, x.shape, x.dtype.str)

        wl = W.prefill(T=T)
        pspecs = tuple(put(wl[n]) for n in ("q", "k", "v", "a", "dt_bias", "A_log", "b", "h0"))
        H = wl["H"]
        self.prefill_tasks = [(pspecs, list(range(H))[i::self.cores], wl["scale"])
                              for i in range(min(self.cores, H))]
        self.decode_tasks = []
        self.decode_rows = 0
        if with_decode:
            dw = W.decode()
            dspecs = tuple(put(dw[n]) for n in ("packed_qkv", "a", "b", "A_log", "dt_bias", "state_pool", "indices"))
            dims = dict(H=dw["H"], HV=dw["HV"], K=dw["K"], V=dw["V"], scale=dw["scale"])
            idx = dw["indices"].tolist()
            for i in range(self.cores):
                rows = list(range(dw["B"]))[i::self.cores]
                if not rows:
                    continue
                local, j = [], 0
                for r in rows:  # slots renumbered over the rows' compacted pool
                    local.append(j if idx[r] >= 0 else -1)
                    j += idx[r] >= 0
                self.decode_tasks.append((dspecs, rows, np.array(local), dims))
                self.decode_rows += len(rows)
            del dw
        del wl
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_pool_init)

    def prefill_seconds(self):
        t0 = time.perf_counter()
        self.pool.map(_oracle_prefill_part, self.prefill_tasks, chunksize=1)
        return time.perf_counter() - t0

    def decode_seconds(self):
        if not self.decode_tasks:
            return 0.0
        t0 = time.perf_counter()
        self.pool.map(_oracle_decode_part, self.decode_tasks, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()
        for shm in self._shm:
            shm.close()
            shm.unlink()
        self._shm = []


def oracle_parallel_baseline(budget_s=20.0):
    """cpu_baseline: the token-recurrence oracle on all host cores over the full
    prefill (all 8192 tokens, all 32 heads), or its first tokens if one run would
    exceed budget_s. Returns (tokens/s, sample text, cores)."""
    cores = int(os.cpu_count() or 1)
    T = PREFILL_T
    # calibrate on 64 tokens in parallel, then size the run to the budget
    cal = OracleCpu(T=64, cores=cores, with_decode=False)
    try:
        cal.prefill_seconds()  # warm the workers (imports)
        per_tok = cal.prefill_seconds() / 64
    finally:
        cal.close()
    T = int(max(256, min(PREFILL_T, budget_s / max(per_tok, 1e-9))))
    T -= T % 16
    oc = OracleCpu(T=T, cores=cores, with_decode=False)
    try:
        oc.prefill_seconds()
        dt = oc.prefill_seconds()
    finally:
        oc.close()
    sample = (f"fp64 token-recurrence oracle, first {T} of 8192 tokens of the prefill workload, all 32 heads "
              f"split over {cores} worker processes (one per host core, one thread each), {dt:.2f} s wall")
    return T / dt, sample, cores


def oracle_sample(T_sample=None, budget_s=20.0, chunk_size=None):
    """Time the fp64 oracle (as it stands: the token recurrence, or with
    chunk_size its chunked form) on the first tokens of the prefill workload,
    all 32 heads. Returns (tokens/s, sample text, cores)."""
    import numpy as np  # noqa: F401

    from kimi_delta_attention_04_gb300 import workloads as W
    from oracle import kda_oracle as ko

    wl = W.prefill()
    np64 = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    # calibrate on 32 tokens, then size the sample to the time budget
    T_cal = 32
    t0 = time.perf_counter()
    ko.kda_forward(np64(wl["q"][:, :T_cal]), np64(wl["k"][:, :T_cal]), np64(wl["v"][:, :T_cal]),
                   scale=wl["scale"], a=np64(wl["a"][:, :T_cal]), dt_bias=np64(wl["dt_bias"]),
                   A_log=np64(wl["A_log"]), b=np64(wl["b"][:, :T_cal]), h0=np64(wl["h0"]), l2norm_qk=True,
                   chunk_size=chunk_size)
    per_tok = (time.perf_counter() - t0) / T_cal
    if T_sample is None:
        T_sample = int(max(64, min(PREFILL_T, budget_s / max(per_tok, 1e-6))))
    t0 = time.perf_counter()
    ko.kda_forward(np64(wl["q"][:, :T_sample]), np64(wl["k"][:, :T_sample]), np64(wl["v"][:, :T_sample]),
                   scale=wl["scale"], a=np64(wl["a"][:, :T_sample]), dt_bias=np64(wl["dt_bias"]),
                   A_log=np64(wl["A_log"]), b=np64(wl["b"][:, :T_sample]), h0=np64(wl["h0"]), l2norm_qk=True,
                   chunk_size=chunk_size)
    dt = time.perf_counter() - t0
    form = "token-recurrence" if chunk_size is None else f"chunked (C={chunk_size})"
    sample = (f"fp64 {form} oracle, first {T_sample} of 8192 tokens of the prefill workload, "
              f"all 32 heads, one process ({dt:.1f} s)")
    return T_sample / dt, sample, 1


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, on the host cores of this
    machine, timing whole steps of the same workload (one full prefill forward
    and one full decode step per step), with the GPU arm's config."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    T = args.ref_seq_len
    oc = OracleCpu(T=T)
    try:
        oc.prefill_seconds()  # start the workers, import and attach the inputs (not timed)
        oc.decode_seconds()
        pre, dec = [], []
        for i in range(args.warmup + args.steps):
            tp = oc.prefill_seconds()
            td = oc.decode_seconds()
            if i >= args.warmup:
                pre.append(tp)
                dec.append(td)
    finally:
        oc.close()
    t_pre = statistics.median(pre)
    value = T / t_pre
    step_ms = [1000.0 * (a + b) for a, b in zip(pre, dec)]
    sample = (f"whole steps: the fp64 token-recurrence oracle over {T} of 8192 tokens x 32 heads of the prefill, "
              f"then the fp64 decode oracle over all {oc.decode_rows} rows, split over {oc.cores} worker "
              f"processes (one per host core, one thread each)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(world),
        "reference": {"what": "fp64 CPU oracle (oracle/kda_oracle.py) as it stands", "timed": "every step",
                      "prefill_s_median": t_pre, "decode_us_per_step": 1e6 * statistics.median(dec)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oc.cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if T != PREFILL_T:
        line["config"]["partial"] = f"ref_seq_len={T}: a test run, not the benchmark line"
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from kimi_delta_attention_04_gb300 import build as kbuild
    kbuild.build()
    import kimi_delta_attention_04_gb300 as kda
    from kimi_delta_attention_04_gb300 import workloads as W

    stream = torch.cuda.current_stream(dev)
    # --- inputs (replica per rank: seeds differ, shapes identical) ---
    T = args.seq_len
    wl = W.prefill(seed=2 + 100 * rank, T=T)
    dw = W.decode(seed=4 + 100 * rank) if args.only in ("all", "decode") else W.decode(seed=4, B=8, num_slots=16)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in wl.items()}
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in dw.items()}
    o = torch.empty(1, T, PREFILL_H, D, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(1, PREFILL_H, D, D, dtype=torch.float32, device=dev)
    args_c = kda.make_chunk_args(d["q"], d["k"], d["v"], scale=d["scale"], a=d["a"], dt_bias=d["dt_bias"],
                                 A_log=d["A_log"], b=d["b"], h0=d["h0"], l2norm_qk=True, o=o, hT=hT)
    ws = torch.empty(kda.chunk_workspace_size(args_c), dtype=torch.uint8, device=dev)
    pool = dd["state_pool"]
    od = torch.empty(dw["B"], dw["HV"], dw["V"], dtype=torch.bfloat16, device=dev)
    n_valid = int((dw["indices"] >= 0).sum())

    def chunk_step():
        if args.only not in ("all", "chunk"):
            return
        kda.kda_chunk_fwd(d["q"], d["k"], d["v"], scale=d["scale"], a=d["a"], dt_bias=d["dt_bias"],
                          A_log=d["A_log"], b=d["b"], h0=d["h0"], l2norm_qk=True, o=o, hT=hT, workspace=ws,
                          stream=stream)

    def decode_step():
        if args.only not in ("all", "decode"):
            return
        kda.kda_decode_step(dd["packed_qkv"], dd["a"], dd["b"], dd["A_log"], dd["dt_bias"], pool, dd["indices"],
                            H=dw["H"], HV=dw["HV"], K=dw["K"], V=dw["V"], scale=dw["scale"], o=od, stream=stream)

    for _ in range(args.warmup):
        chunk_step()
        decode_step()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clocks:
        e0.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            chunk_step()
            ev[i][1].record(stream)
            decode_step()
            ev[i][2].record(stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    chunk_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    total_ms = e0.elapsed_time(e1)

    # --- decode launch overheads: host wall-clock per step including the launch,
    # and the same steps replayed from a CUDA graph ---
    dec_wall = dec_graph = None
    if args.only in ("all", "decode"):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(K):
            decode_step()
        torch.cuda.synchronize(dev)
        dec_wall = (time.perf_counter() - t0) / K
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                kda.kda_decode_step(dd["packed_qkv"], dd["a"], dd["b"], dd["A_log"], dd["dt_bias"], pool,
                                    dd["indices"], H=dw["H"], HV=dw["HV"], K=dw["K"], V=dw["V"], scale=dw["scale"],
                                    o=od, stream=cap)
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(K):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        dec_graph = g0.elapsed_time(g1) / 1000.0 / K

    # --- e2e through the public API with pinned host buffers: every step copies
    # its inputs in from pinned host memory and reads o and hT back. The copies run
    # on their own streams with two device buffers each way, so step i+1's inputs
    # travel while step i computes and step i-1's outputs travel back. ---
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in wl.items()}
    names = ("q", "k", "v", "a", "dt_bias", "A_log", "b", "h0")
    o_hs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hT_hs = [torch.empty(hT.shape, dtype=hT.dtype).pin_memory() for _ in range(2)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_hs[0].numel() * o_hs[0].element_size() + hT_hs[0].numel() * hT_hs[0].element_size()
    e2e_steps = max(4, min(K, 10)) if args.only in ("all", "chunk") else 0
    e2e_s = 0.0
    if e2e_steps:
        h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        dbuf = [{n: torch.empty_like(host[n], device=dev) for n in names} for _ in range(2)]
        obuf = [torch.empty_like(o) for _ in range(2)]
        hbuf = [torch.empty_like(hT) for _ in range(2)]
        in_ready, in_free, out_ready, out_free = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            sl = i % 2
            with torch.cuda.stream(h2d_stream):
                if i >= 2:
                    h2d_stream.wait_event(in_free[sl])
                for n in names:
                    dbuf[sl][n].copy_(host[n], non_blocking=True)
                in_ready[sl].record(h2d_stream)
            stream.wait_event(in_ready[sl])
            if i >= 2:
                stream.wait_event(out_free[sl])
            di = dbuf[sl]
            kda.kda_chunk_fwd(di["q"], di["k"], di["v"], scale=wl["scale"], a=di["a"], dt_bias=di["dt_bias"],
                              A_log=di["A_log"], b=di["b"], h0=di["h0"], l2norm_qk=True, o=obuf[sl], hT=hbuf[sl],
                              workspace=ws, stream=stream)
            in_free[sl].record(stream)
            out_ready[sl].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(out_ready[sl])
                o_hs[sl].copy_(obuf[sl], non_blocking=True)
                hT_hs[sl].copy_(hbuf[sl], non_blocking=True)
                out_free[sl].record(d2h_stream)
        torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - t0) / e2e_steps

    # --- varlen prefill: 16 packed sequences (its own timed region) ---
    var = None
    if args.only == "all":
        vw = W.varlen(seed=3 + 100 * rank)
        vd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in vw.items()}
        n_seq = int(vd["cu_seqlens"].numel()) - 1
        t_tot = int(vw["q"].shape[1])
        vo = torch.empty_like(vd["v"])
        vhT = torch.empty(n_seq, PREFILL_H, D, D, dtype=torch.float32, device=dev)
        vargs = kda.make_chunk_args(vd["q"], vd["k"], vd["v"], scale=vd["scale"], a=vd["a"], dt_bias=vd["dt_bias"],
                                    A_log=vd["A_log"], b=vd["b"], h0=vd["h0"], cu_seqlens=vd["cu_seqlens"],
                                    l2norm_qk=True, o=vo, hT=vhT)
        vws = torch.empty(kda.chunk_workspace_size(vargs), dtype=torch.uint8, device=dev)

        def var_step():
            kda.kda_chunk_fwd(vd["q"], vd["k"], vd["v"], scale=vd["scale"], a=vd["a"], dt_bias=vd["dt_bias"],
                              A_log=vd["A_log"], b=vd["b"], h0=vd["h0"], cu_seqlens=vd["cu_seqlens"],
                              l2norm_qk=True, o=vo, hT=vhT, workspace=vws, stream=stream)
        for _ in range(args.warmup):
            var_step()
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        v0.record(stream)
        for _ in range(K):
            var_step()
        v1.record(stream)
        torch.cuda.synchronize(dev)
        v_avg = v0.elapsed_time(v1) / 1000.0 / K
        vbytes = t_tot * BYTES_PER_TOKEN + 2 * n_seq * STATE_BYTES + PARAM_BYTES
        var = {"ms": 1000.0 * v_avg, "sequences": n_seq, "tokens": t_tot, "tokens_per_s": t_tot / v_avg,
               "algorithmic_bytes": vbytes, "achieved_gbs": vbytes / v_avg / 1e9,
               "launches_per_call": 2, "note": "kda_plan_kernel + kda_chunk_fused_kernel"}

    # --- the prefill with the log-decay g given (fp32 [1, T, 32, 128], KDA_GATE_G;
    # drawn directly, same bytes as the gate inputs a): its own timed region ---
    gate_g = None
    if args.only == "all":
        gw = W.prefill(seed=7 + 100 * rank, T=T, gate="g")
        gd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in gw.items()}
        go = torch.empty_like(o)
        ghT = torch.empty_like(hT)

        def g_step():
            kda.kda_chunk_fwd(gd["q"], gd["k"], gd["v"], scale=gd["scale"], g=gd["g"], b=gd["b"], h0=gd["h0"],
                              l2norm_qk=True, o=go, hT=ghT, workspace=ws, stream=stream)
        for _ in range(args.warmup):
            g_step()
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        q0.record(stream)
        for _ in range(K):
            g_step()
        q1.record(stream)
        torch.cuda.synchronize(dev)
        g_avg = q0.elapsed_time(q1) / 1000.0 / K
        gbytes = prefill_algorithmic_bytes(T) - PARAM_BYTES
        gate_g = {"ms": 1000.0 * g_avg, "tokens_per_s": T / g_avg, "algorithmic_bytes": gbytes,
                  "achieved_gbs": gbytes / g_avg / 1e9, "kernel": "kda_chunk_fused_kernel (KDA_GATE_G)",
                  "inputs": "g = -U(0.01, 3) fp32 drawn directly (one exp per element in the kernel instead of "
                            "the gate's exp, log and exp)"}
        del gd, gw

    # --- decode with the causal conv1d + SiLU fused in front (its own timed region) ---
    dconv = None
    if args.only == "all":
        cw = W.decode_conv_workload(seed=6 + 100 * rank, W=4)
        cd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in cw.items()}
        oc = torch.empty(cw["B"], cw["HV"], cw["V"], dtype=torch.bfloat16, device=dev)

        def conv_step():
            kda.kda_decode_conv_step(cd["packed_qkv"], cd["conv_state"], cd["conv_weight"], cd["conv_bias"], cd["a"],
                                     cd["b"], cd["A_log"], cd["dt_bias"], cd["state_pool"], cd["indices"], H=cw["H"],
                                     HV=cw["HV"], K=cw["K"], V=cw["V"], scale=cw["scale"], o=oc, stream=stream)
        for _ in range(args.warmup):
            conv_step()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        c0.record(stream)
        for _ in range(K):
            conv_step()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        c_avg = c0.elapsed_time(c1) / 1000.0 / K
        c_valid = int((cw["indices"] >= 0).sum())
        C = cw["packed_qkv"].shape[1]
        cbytes = decode_algorithmic_bytes(c_valid) + c_valid * (cw["W"] - 1) * C * 2 * 2 + C * cw["W"] * 4 + C * 4
        dconv = {"us_per_step": 1e6 * c_avg, "width": cw["W"], "n_valid_rows": c_valid, "algorithmic_bytes": cbytes,
                 "achieved_gbs": cbytes / c_avg / 1e9, "kernel": "kda_decode_kernel<conv>"}

    # --- output-side per-head RMSNorm of the prefill's o (its own timed region) ---
    rms = None
    if args.only == "all":
        w_rms = torch.linspace(0.5, 1.5, D, device=dev)
        y_rms = torch.empty_like(o)
        for _ in range(args.warmup):
            kda.kda_head_rmsnorm(o, w_rms, eps=1e-6, out=y_rms, stream=stream)
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        n0.record(stream)
        for _ in range(K):
            kda.kda_head_rmsnorm(o, w_rms, eps=1e-6, out=y_rms, stream=stream)
        n1.record(stream)
        torch.cuda.synchronize(dev)
        n_avg = n0.elapsed_time(n1) / 1000.0 / K
        nbytes = 2 * o.numel() * o.element_size() + D * 4
        rms = {"us": 1e6 * n_avg, "rows": o.numel() // D, "algorithmic_bytes": nbytes,
               "achieved_gbs": nbytes / n_avg / 1e9, "kernel": "kda_rmsnorm_kernel",
               "note": "64 MB in + 64 MB out: partly served by L2 (129 MB), so it can exceed the HBM copy rate"}

    # --- short-T recurrent step (its own timed regions, not part of the step) ---
    def recurrent_field(B_r, T_r, slots):
        rw = W.recurrent_workload(seed=5 + 100 * rank, B=B_r, T=T_r, num_slots=slots)
        rd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in rw.items()}
        orr = torch.empty(rw["B"], rw["T"], rw["HV"], rw["V"], dtype=torch.bfloat16, device=dev)

        def rec_step():
            kda.kda_recurrent_step(rd["q"], rd["k"], rd["v"], rd["a"], rd["b"], rd["A_log"], rd["dt_bias"],
                                   rd["state_pool"], rd["indices"], scale=rw["scale"], o=orr, stream=stream)
        for _ in range(args.warmup):
            rec_step()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        r0.record(stream)
        for _ in range(K):
            rec_step()
        r1.record(stream)
        torch.cuda.synchronize(dev)
        r_avg = r0.elapsed_time(r1) / 1000.0 / K
        r_valid = int((rw["indices"] >= 0).sum())
        rbytes = recurrent_algorithmic_bytes(r_valid, rw["B"], rw["T"])
        kernel = "kda_recurrent_tc_kernel (chunk form, tensor cores)" if T_r >= 8 else "kda_recurrent_kernel (per token)"
        # the stored DRAM traffic was captured at 128 rows x 8 tokens and at 64 rows x 64
        # tokens (the instance that keeps the state in tensor memory between chunks); at a
        # given T it scales by the valid rows (the slots dominate)
        rsha = kernel_sources_sha(RECURRENT_KERNEL_SOURCES)
        traffic = (stored_traffic("kda_recurrent_tc_kernel", rsha, r_valid) if T_r == RECURRENT_T else
                   stored_traffic("kda_recurrent_tc_kernel_T64", rsha, r_valid) if T_r == RECURRENT_LONG_T else None)
        return {"us_per_step": 1e6 * r_avg, "rows": rw["B"], "tokens_per_row": rw["T"], "n_valid_rows": r_valid,
                "tokens_per_s": rw["B"] * rw["T"] / r_avg,
                "roofline": {"bound": "hbm", "achieved": rbytes / r_avg / 1e9, "unit": "GB/s",
                             "algorithmic_bytes": rbytes, "kernel": kernel, "traffic": traffic}}

    rec = rec_long = None
    if args.only in ("all", "recurrent"):
        rec = recurrent_field(RECURRENT_B, RECURRENT_T, RECURRENT_SLOTS)
        rec_long = recurrent_field(RECURRENT_LONG_B, RECURRENT_LONG_T, 2 * RECURRENT_LONG_B)

    # --- per-chunk entering states, then the chunk-parallel output pass (own timed regions) ---
    cst = None
    if args.only == "all":
        nc = kda.chunk_count(1, T)
        hc = torch.empty(nc, PREFILL_H, D, D, dtype=torch.float32, device=dev)
        o_par = torch.empty_like(o)
        sargs = kda.make_chunk_args(d["q"], d["k"], d["v"], scale=d["scale"], a=d["a"], dt_bias=d["dt_bias"],
                                    A_log=d["A_log"], b=d["b"], h0=d["h0"], l2norm_qk=True, o=o, hT=hT, h_chunks=hc)
        sws = torch.empty(kda.chunk_workspace_size(sargs), dtype=torch.uint8, device=dev)

        def snap_step():
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], scale=d["scale"], a=d["a"], dt_bias=d["dt_bias"],
                              A_log=d["A_log"], b=d["b"], h0=d["h0"], l2norm_qk=True, o=o, hT=hT, workspace=sws,
                              h_chunks=hc, stream=stream)

        def par_step():
            kda.kda_chunk_output(d["q"], d["k"], d["v"], hc, scale=d["scale"], a=d["a"], dt_bias=d["dt_bias"],
                                 A_log=d["A_log"], b=d["b"], l2norm_qk=True, o=o_par, workspace=sws, stream=stream)

        def timed(fn):
            for _ in range(args.warmup):
                fn()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            s0.record(stream)
            for _ in range(K):
                fn()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            return s0.elapsed_time(s1) / 1000.0 / K
        t_snap = timed(snap_step)
        t_par = timed(par_step)
        hc_bytes = hc.numel() * 4
        snap_bytes = prefill_algorithmic_bytes(T) + hc_bytes
        par_bytes = T * BYTES_PER_TOKEN + PARAM_BYTES + hc_bytes
        cst = {"chunks": nc, "h_chunks_bytes": hc_bytes,
               "fwd_with_states": {"ms": 1000.0 * t_snap, "algorithmic_bytes": snap_bytes,
                                   "achieved_gbs": snap_bytes / t_snap / 1e9,
                                   "kernel": "kda_chunk_fused_kernel (its recurrence writes h_chunks)"},
               "output_pass": {"ms": 1000.0 * t_par, "algorithmic_bytes": par_bytes,
                               "achieved_gbs": par_bytes / t_par / 1e9,
                               "kernel": "kda_chunk_fused_kernel, output-pass mode (state of each chunk read from h_chunks)"}}

    # --- reduce over ranks: max time ---
    t_chunk = sum(chunk_ms) / 1000.0
    t_dec = sum(dec_ms) / 1000.0
    t_total = total_ms / 1000.0
    t_chunk, t_dec, t_total, e2e_s = max_over_ranks([t_chunk, t_dec, t_total, e2e_s], dev)
    tokens = T * K * world
    value = tokens / t_chunk if t_chunk > 0 else 0.0

    hbm, tflops, peak_kind = load_peaks()
    chunk_avg = t_chunk / K
    dec_avg = t_dec / K
    abytes = prefill_algorithmic_bytes(T)
    aflops = prefill_algorithmic_flops(T)
    achieved = abytes / chunk_avg / 1e9 if chunk_avg > 0 else 0.0
    t_roof = max(abytes / (hbm * 1e9), aflops / (tflops * 1e12))
    dbytes = decode_algorithmic_bytes(n_valid)
    dach = dbytes / dec_avg / 1e9 if dec_avg > 0 else 0.0
    chunk_sha = kernel_sources_sha(CHUNK_KERNEL_SOURCES)
    dec_sha = kernel_sources_sha(DECODE_KERNEL_SOURCES)
    clk = clocks.summary()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t_total / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": bench_config(world),
            "chunk_fwd": {"ms": 1000.0 * chunk_avg, "tokens_per_s": value,
                          "roofline_time_us": 1e6 * t_roof, "frac_of_roofline": t_roof / chunk_avg if chunk_avg > 0 else 0.0},
            "varlen": var,
            "prefill_gate_g": gate_g,
            "head_rmsnorm": rms,
            "decode_conv": dconv,
            "recurrent": rec,
            "recurrent_long": rec_long,
            "chunk_states": cst,
            "decode": {"us_per_step": 1e6 * dec_avg, "n_valid_rows": n_valid,
                       "wall_us_per_step_with_launch": None if dec_wall is None else 1e6 * dec_wall,
                       "graph_replay_us_per_step": None if dec_graph is None else 1e6 * dec_graph,
                       "roofline": {"bound": "hbm", "achieved": dach, "peak": hbm, "unit": "GB/s",
                                    "frac": dach / hbm, "frac_of_spec_peak": dach / SPEC_HBM_GBS,
                                    "spec_peak": SPEC_HBM_GBS, "algorithmic_bytes": dbytes,
                                    "traffic": stored_traffic("kda_decode_kernel", dec_sha, n_valid), "peak_kind": peak_kind}},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "frac_of_spec_peak": achieved / SPEC_HBM_GBS, "spec_peak": SPEC_HBM_GBS,
                         "traffic": stored_traffic("kda_chunk_fused_kernel", chunk_sha, T), "kernel": "kda_chunk_fused_kernel (prep + recurrence in one launch)",
                         "algorithmic_bytes": abytes, "peak_kind": peak_kind},
            "e2e": {"value": T * world / e2e_s if e2e_steps else None, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "note": "copies on their own streams, two buffers each way: step i+1's inputs in and step "
                            "i-1's o and hT out while step i computes"},
            "gpu_launches": (CHUNK_LAUNCHES_PER_STEP if args.only in ("all", "chunk") else 0) * K
                            + (DECODE_LAUNCHES_PER_STEP if args.only in ("all", "decode") else 0) * K,
            "clocks": clk,
        }
        if var is not None:
            var["frac_of_roofline"] = var["achieved_gbs"] / hbm
            var["frac_of_spec_peak"] = var["achieved_gbs"] / SPEC_HBM_GBS
        if gate_g is not None:
            gate_g["frac_of_roofline"] = gate_g["achieved_gbs"] / hbm
        if rms is not None:
            rms["frac_of_hbm"] = rms["achieved_gbs"] / hbm
        if dconv is not None:
            dconv["frac_of_hbm"] = dconv["achieved_gbs"] / hbm
        if cst is not None:
            for part in ("fwd_with_states", "output_pass"):
                cst[part]["frac_of_hbm"] = cst[part]["achieved_gbs"] / hbm
        for r in (rec, rec_long):
            if r is not None:
                r["roofline"]["peak"] = hbm
                r["roofline"]["frac"] = r["roofline"]["achieved"] / hbm
                r["roofline"]["peak_kind"] = peak_kind
        if args.only != "all" or T != PREFILL_T:
            line["config"]["partial"] = f"only={args.only}, seq_len={T}: a profiling run, not the benchmark line"
        # a leg that did not run reports nothing (its events bracket an empty region)
        if args.only not in ("all", "chunk"):
            line["value"] = None
            line["chunk_fwd"] = None
            line["roofline"] = None
        if args.only not in ("all", "decode"):
            line["decode"] = None
        if world == 1 and not args.no_cpu_baseline:
            v, sample, cores = oracle_parallel_baseline(budget_s=args.cpu_budget)
            line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
            v, sample, cores = oracle_sample(budget_s=args.cpu_budget / 3)
            line["cpu_baseline_1core"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                          "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seq-len", type=int, default=PREFILL_T,
                    help="prefill tokens of each --impl reference step (tests use fewer; the line is then partial)")
    ap.add_argument("--only", choices=["all", "chunk", "decode", "recurrent"], default="all",
                    help="time only one part (profiling runs; the benchmark line uses all)")
    ap.add_argument("--seq-len", type=int, default=PREFILL_T, help="prefill tokens (profiling runs use fewer)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
