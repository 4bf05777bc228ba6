"""Per-chunk entering states (h_chunks) written by kda_chunk_fwd and the
chunk-parallel output pass kda_chunk_output, against the fp64 oracle through
the C ABI: snapshots, o and hT within the bf16 tolerances (rel-Frobenius
<= 5e-3, max-abs <= 2e-2)."""

import pytest
import torch

import kimi_delta_attention_04_gb300 as kda
from kimi_delta_attention_04_gb300 import workloads as W
from oracle import kda_oracle as ko

from kda_cases import Canary, assert_close, np64, subset_heads, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_04_gb300 import build
    build.build()
    kda.load()


def _kw(d):
    return dict(scale=d["scale"], g=d["g"], a=d["a"], dt_bias=d["dt_bias"], A_log=d["A_log"], beta=d["beta"],
                b=d["b"], cu_seqlens=d["cu_seqlens"], l2norm_qk=d["l2norm"], delta=d["delta"], g_head=d.get("g_head"))


@pytest.mark.parametrize("K,B,T,lengths,gate", [
    (64, 2, 70, None, "inputs"),
    (128, 1, 200, None, "inputs"),
    (128, 1, 0, [40, 0, 130, 17], "inputs"),
    (128, 2, 45, None, "head"),
], ids=["d64", "d128", "d128_varlen", "d128_gdn"])
def test_chunk_states_and_parallel_output(K, B, T, lengths, gate):
    wl = W.chunk_workload(seed=140 + K + (T or 7), B=B, T=T or 1, H=3, K=K, V=K, lengths=lengths, gate=gate)
    d = to_dev(wl)
    nc = kda.chunk_count(wl["B"], wl["T"], wl["cu_seqlens"])
    cn = Canary()
    hc = cn.empty((nc, wl["H"], K, K), torch.float32, name="h_chunks")
    hc.fill_(float("nan"))
    o = cn.empty(tuple(d["q"].shape[:3]) + (K,), torch.bfloat16, name="o")
    hT = cn.empty((wl["N"], wl["H"], K, K), torch.float32, name="hT")
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], h0=d["h0"], h_chunks=hc, o=o, hT=hT, **_kw(d))
    cn.check()
    o_ref, h_ref, s_ref = ko.kda_forward(
        np64(wl["q"]), np64(wl["k"]), np64(wl["v"]), scale=wl["scale"], g=np64(wl["g"]), a=np64(wl["a"]),
        dt_bias=np64(wl["dt_bias"]), A_log=np64(wl["A_log"]), beta=np64(wl["beta"]), b=np64(wl["b"]),
        h0=np64(wl["h0"]), cu_seqlens=None if wl["cu_seqlens"] is None else wl["cu_seqlens"].numpy(),
        l2norm_qk=wl["l2norm"], delta=wl["delta"], g_head=np64(wl.get("g_head")), chunk_states=True)
    assert s_ref.shape[0] == nc
    assert_close("snapshots", np64(hc), s_ref, torch.bfloat16)
    assert_close("o (snapshot path)", np64(o), o_ref, torch.bfloat16)
    assert_close("hT (snapshot path)", np64(hT), h_ref, torch.bfloat16)
    # every chunk's output again, in parallel, from its snapshot
    o2 = cn.empty(tuple(o.shape), torch.bfloat16, name="o (output pass)")
    kda.kda_chunk_output(d["q"], d["k"], d["v"], hc, o=o2, **_kw(d))
    cn.check()
    assert_close("o (chunk-parallel pass)", np64(o2), o_ref, torch.bfloat16)


def test_chunk_states_noalloc_matches_workspace_call():
    """The no-alloc entry point with per-chunk states writes the same states and o."""
    wl = W.chunk_workload(seed=151, B=1, T=90, H=2, K=128, V=128)
    d = to_dev(wl)
    nc = kda.chunk_count(1, 90)
    hc1 = torch.zeros(nc, 2, 128, 128, dtype=torch.float32, device="cuda")
    hc2 = torch.ones_like(hc1)
    o1, h1 = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], h0=d["h0"], h_chunks=hc1, **_kw(d))
    o2, h2 = kda.kda_chunk_fwd_noalloc(d["q"], d["k"], d["v"], h0=d["h0"], h_chunks=hc2, **_kw(d))
    torch.cuda.synchronize()
    assert torch.equal(hc1, hc2)
    assert torch.equal(o1, o2)
    assert torch.equal(h1, h2)


def test_chunk_states_full_size_sampled_heads():
    """The prefill recipe at full size (B=1, H=32, T=8192) in the benchmark's
    launch: the fused kernel's snapshot forward and output pass; the oracle
    recomputes the per-chunk states and o of two heads (heads are independent),
    and the output pass must give the forward's o."""
    wl = W.prefill()
    d = to_dev(wl)
    nc = kda.chunk_count(1, wl["T"])
    cn = Canary()
    hc = cn.empty((nc, wl["H"], 128, 128), torch.float32, name="h_chunks")
    o = cn.empty((1, wl["T"], wl["H"], 128), torch.bfloat16, name="o")
    hT = cn.empty((1, wl["H"], 128, 128), torch.float32, name="hT")
    o2 = cn.empty((1, wl["T"], wl["H"], 128), torch.bfloat16, name="o (output pass)")
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], h0=d["h0"], h_chunks=hc, o=o, hT=hT, **_kw(d))
    kda.kda_chunk_output(d["q"], d["k"], d["v"], hc, o=o2, **_kw(d))
    o_plain, _ = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], h0=d["h0"], **_kw(d))
    cn.check()
    assert_close("snapshot forward vs plain forward", np64(o), np64(o_plain), torch.bfloat16)
    heads = [2, 29]
    sub = subset_heads(wl, heads)
    o_ref, h_ref, s_ref = ko.kda_forward(
        np64(sub["q"]), np64(sub["k"]), np64(sub["v"]), scale=sub["scale"], a=np64(sub["a"]),
        dt_bias=np64(sub["dt_bias"]), A_log=np64(sub["A_log"]), b=np64(sub["b"]), h0=np64(sub["h0"]),
        l2norm_qk=sub["l2norm"], delta=sub["delta"], chunk_states=True)
    assert_close("full snapshots", np64(hc[:, heads]), s_ref, torch.bfloat16)
    assert_close("full o (snapshot forward)", np64(o)[:, :, heads], o_ref, torch.bfloat16)
    assert_close("full hT (snapshot forward)", np64(hT)[:, heads], h_ref, torch.bfloat16)
    assert_close("full o (output pass)", np64(o2)[:, :, heads], o_ref, torch.bfloat16)
    assert_close("output pass vs forward", np64(o2), np64(o), torch.bfloat16)
