"""Helpers shared by the GPU parity tests: run a workload through the CUDA
path (libkda via the Python binding) and through the fp64 oracle, and compare.

Inputs come only from kimi_delta_attention_04_gb300.workloads; expected values
only from oracle/."""

from __future__ import annotations

import numpy as np
import torch

import kimi_delta_attention_04_gb300 as kda
from oracle import kda_oracle as ko

BF16_REL_F = 5e-3   # relative Frobenius error of o and hT, bf16 inputs
BF16_MAX_ABS = 2e-2  # max abs error, bf16 inputs
FP32_MAX_ABS = 1e-4  # max abs error, fp32 inputs


GUARD_BYTES = 256   # canary band on each side of an output (a multiple of 16: keeps the output aligned)
SENTINEL = 0xA5     # byte pattern of the bands


class Canary:
    """Output buffers with a band of GUARD_BYTES sentinel bytes on each side.

    compute-sanitizer is not used on this hardware, so the tests catch stores
    that land just outside an output this way: every output a test passes to the
    library comes from here, and check() asserts, after the GPU work, that no
    band byte changed (a ragged tail, a varlen boundary or an empty sequence
    writing one row or one chunk too far would show up)."""

    def __init__(self):
        self._bufs = []

    def empty(self, shape, dtype, device="cuda", name="out"):
        el = torch.empty((), dtype=dtype).element_size()
        n = 1
        for x in shape:
            n *= int(x)
        pad = GUARD_BYTES // el
        buf = torch.empty(n + 2 * pad, dtype=dtype, device=device)
        buf.view(torch.uint8).fill_(SENTINEL)
        self._bufs.append((name, buf, n * el))
        return buf[pad:pad + n].view(*shape)

    def clone(self, src, name="out"):
        t = self.empty(tuple(src.shape), src.dtype, src.device, name)
        t.copy_(src)
        return t

    def check(self):
        torch.cuda.synchronize()
        for name, buf, nbytes in self._bufs:
            raw = buf.view(torch.uint8)
            lo, hi = raw[:GUARD_BYTES], raw[GUARD_BYTES + nbytes:]
            assert hi.numel() == GUARD_BYTES
            assert bool((lo == SENTINEL).all()), f"{name}: bytes written before the start of the output"
            assert bool((hi == SENTINEL).all()), f"{name}: bytes written past the end of the output"


def np64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def to_dev(wl, device="cuda"):
    out = dict(wl)
    for key in ("q", "k", "v", "g", "g_head", "a", "dt_bias", "A_log", "beta", "b", "h0", "cu_seqlens"):
        if out.get(key) is not None:
            out[key] = out[key].to(device).contiguous()
    return out


def gpu_chunk(wl, *, h0=True, final_state=True, err=None, workspace=None, o=None, hT=None):
    """The chunk forward through the C ABI. Outputs the caller does not pass come
    with canary bands, checked (after a synchronize) before returning."""
    d = to_dev(wl)
    cn = Canary()
    N = (d["cu_seqlens"].numel() - 1) if d["cu_seqlens"] is not None else d["q"].shape[0]
    if o is None:
        o = cn.empty(tuple(d["q"].shape[:3]) + (d["v"].shape[-1],), d["q"].dtype, name="o")
    if hT is None and final_state:
        hT = cn.empty((N, d["q"].shape[2], d["v"].shape[-1], d["q"].shape[-1]), torch.float32, name="hT")
    out = kda.kda_chunk_fwd(
        d["q"], d["k"], d["v"], scale=d["scale"], g=d["g"], a=d["a"], dt_bias=d["dt_bias"], A_log=d["A_log"],
        beta=d["beta"], b=d["b"], h0=d["h0"] if h0 else None, cu_seqlens=d["cu_seqlens"],
        l2norm_qk=d["l2norm"], delta=d["delta"], output_final_state=final_state, err=err, workspace=workspace,
        o=o, hT=hT, g_head=d.get("g_head"))
    cn.check()
    return out


def oracle_chunk(wl, *, h0=True, chunk_size=None):
    return ko.kda_forward(
        np64(wl["q"]), np64(wl["k"]), np64(wl["v"]), scale=wl["scale"], g=np64(wl["g"]), a=np64(wl["a"]),
        dt_bias=np64(wl["dt_bias"]), A_log=np64(wl["A_log"]), beta=np64(wl["beta"]), b=np64(wl["b"]),
        h0=np64(wl["h0"]) if h0 else None, cu_seqlens=None if wl["cu_seqlens"] is None else wl["cu_seqlens"].numpy(),
        l2norm_qk=wl["l2norm"], delta=wl["delta"], chunk_size=chunk_size, g_head=np64(wl.get("g_head")))


def subset_heads(wl, heads):
    """The same workload restricted to some heads (heads are independent)."""
    heads = list(heads)
    K = wl["K"]
    out = dict(wl)
    out["H"] = len(heads)
    idx = torch.tensor(heads)
    for key in ("q", "k", "v", "g", "g_head", "beta", "b"):
        if wl.get(key) is not None:
            out[key] = wl[key].index_select(2, idx).contiguous()
    if wl.get("a") is not None:
        B, T = wl["a"].shape[:2]
        out["a"] = wl["a"].view(B, T, wl["H"], K).index_select(2, idx).reshape(B, T, len(heads) * K).contiguous()
        out["dt_bias"] = wl["dt_bias"].view(wl["H"], K).index_select(0, idx).reshape(-1).contiguous()
        out["A_log"] = wl["A_log"].index_select(0, idx).contiguous()
    if wl.get("h0") is not None:
        out["h0"] = wl["h0"].index_select(1, idx).contiguous()
    return out


def subset_sequence(wl, n):
    """Sequence n of a packed (cu_seqlens) workload as a batch of one."""
    cu = wl["cu_seqlens"]
    s, e = int(cu[n]), int(cu[n + 1])
    out = dict(wl)
    out["cu_seqlens"] = None
    out["N"] = 1
    out["T"] = e - s
    for key in ("q", "k", "v", "g", "g_head", "a", "beta", "b"):
        if wl.get(key) is not None:
            out[key] = wl[key][:, s:e].contiguous()
    if wl.get("h0") is not None:
        out["h0"] = wl["h0"][n:n + 1].contiguous()
    return out


def rel_f(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30))


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64)))) if np.size(ref) else 0.0


def assert_close(name, x, ref, dtype):
    if np.size(ref) == 0:
        return
    ma = max_abs(x, ref)
    if dtype == torch.float32:
        assert ma <= FP32_MAX_ABS, f"{name}: max abs {ma:.3e} > {FP32_MAX_ABS}"
    else:
        rf = rel_f(x, ref)
        assert rf <= BF16_REL_F and ma <= BF16_MAX_ABS, f"{name}: rel-F {rf:.3e}, max abs {ma:.3e}"
