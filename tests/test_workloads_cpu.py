"""The seeded input recipes (kimi_delta_attention_04_gb300/workloads.py): the
sizes, dtypes and value ranges of the benchmark settings, their determinism,
and the padding rule of the slot-pool workloads. CPU only."""

import math

import torch

from kimi_delta_attention_04_gb300 import workloads as W


def test_prefill_recipe_shapes_dtypes_ranges():
    wl = W.prefill(T=256)  # the T=8192 recipe, shortened
    assert wl["q"].shape == (1, 256, 32, 128) and wl["q"].dtype == torch.bfloat16
    assert wl["v"].shape == (1, 256, 32, 128)
    assert wl["a"].shape == (1, 256, 32 * 128) and wl["a"].dtype == torch.float32
    assert wl["dt_bias"].shape == (4096,) and float(wl["dt_bias"].abs().max()) <= 1.0
    assert wl["A_log"].shape == (32,) and 0.0 <= float(wl["A_log"].min()) and float(wl["A_log"].max()) <= 2.0
    assert wl["b"].shape == (1, 256, 32) and wl["b"].dtype == torch.bfloat16
    assert wl["h0"].shape == (1, 32, 128, 128) and wl["h0"].dtype == torch.float32
    assert abs(float(wl["h0"].std()) - 0.1) < 0.01
    assert math.isclose(wl["scale"], 128 ** -0.5)
    assert wl["l2norm"] and wl["delta"]


def test_recipes_are_deterministic_and_seed_dependent():
    a, b, c = W.prefill(T=64), W.prefill(T=64), W.prefill(seed=7, T=64)
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["a"], b["a"]) and torch.equal(a["h0"], b["h0"])
    assert not torch.equal(a["q"], c["q"])


def test_varlen_lengths_recipe():
    lengths = W.varlen_lengths(3)
    assert len(lengths) == 16 and all(512 <= n <= 8192 for n in lengths)
    assert sum(lengths) == 50430  # seed 3, the benchmark's varlen setting
    wl = W.chunk_workload(seed=3, lengths=[5, 0, 17], H=2, K=64, V=64)
    assert wl["cu_seqlens"].tolist() == [0, 5, 5, 22] and wl["B"] == 1 and wl["T"] == 22
    assert wl["h0"].shape == (3, 2, 64, 64)


def test_decode_recipe_padding_and_distinct_slots():
    wl = W.decode()
    idx = wl["indices"]
    assert wl["packed_qkv"].shape == (256, 3 * 32 * 128) and wl["packed_qkv"].dtype == torch.bfloat16
    assert wl["state_pool"].shape == (512, 32, 128, 128)
    assert int((idx < 0).sum()) == 26  # round(0.1 * 256)
    valid = idx[idx >= 0]
    assert len(set(valid.tolist())) == len(valid) and int(valid.max()) < 512


def test_recurrent_and_conv_recipes():
    rw = W.recurrent_workload(B=10, T=3, H=2, HV=4, K=64, V=128, num_slots=20, pad_frac=0.2)
    assert rw["q"].shape == (10, 3, 2, 64) and rw["v"].shape == (10, 3, 4, 128)
    assert rw["a"].shape == (10, 3, 4 * 64) and rw["b"].shape == (10, 3, 4)
    assert int((rw["indices"] < 0).sum()) == 2
    cw = W.decode_conv_workload(B=8, num_slots=16, W=3)
    C = cw["packed_qkv"].shape[1]
    assert cw["conv_state"].shape == (16, 2, C) and cw["conv_weight"].shape == (C, 3)
    assert cw["conv_bias"].shape == (C,)
