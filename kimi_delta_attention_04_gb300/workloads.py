"""Seeded synthetic inputs for the KDA chunk forward and the packed decode.

This module only draws random numbers and casts them to the input dtypes; it
holds none of the method's arithmetic (no gate, no sigmoid, no norm). Both the
CUDA path (through the tests and bench.py) and the fp64 oracle consume what it
returns. Everything is drawn on the CPU with torch.Generator(seed) in a fixed
order, so a workload is reproducible on any machine.

Workloads (the value distributions follow the five benchmark settings of the
KDA chunk forward / decode study):
  fp32_small   fp32, B=1, H=2, T=128, d=64; gate inputs, beta logits, L2 norm
  linear_attn  bf16, B=2, H=4, T=1024, d=128; g = 0, delta off, scale 1
  prefill      bf16, B=1, H=32, T=8192, d=128; gate inputs, beta logits, L2 norm
  varlen       bf16, 16 packed sequences, lengths ~U[512, 8192], H=32, d=128
  decode       B=256, H=HV=32, K=V=128, fp32 pool [512, 32, 128, 128], 10% pads
Smaller variants of the same recipes (fewer tokens, heads or rows) are what the
parity tests use; the recipe and the draw order do not change with the sizes.
"""

from __future__ import annotations

import math

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _randn(gen, shape, dtype, std=1.0):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def _uniform(gen, shape, lo, hi, dtype=torch.float32):
    return (torch.rand(*shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo).to(dtype)


def chunk_workload(*, seed=2, B=1, T=8192, H=32, K=128, V=128, dtype=torch.bfloat16,
                   gate="inputs", beta="logits", l2norm=True, delta=True,
                   A_log_hi=2.0, h0_std=0.1, lengths=None, qkv_std=1.0, scale=None, v_std=None):
    """Inputs of one KDA chunk-forward call.

    Draw order: [lengths], q, k, v, gate inputs (a, dt_bias, A_log) or log-decay g,
    beta logits b or beta, h0. With ``lengths`` the sequences are packed into a
    single row (B = 1) and cu_seqlens is returned.

    gate: "inputs" (a ~ N(0,1) fp32 [B, T, H*K], dt_bias ~ U(-1,1) [H*K],
          A_log ~ U(0, A_log_hi) [H]), "g" (a log-decay g = -U(0.01, 3) fp32
          [B, T, H, K], drawn directly), "head" (Gated DeltaNet: one log-decay
          per token and head, g_head = -U(0.01, 3) fp32 [B, T, H]),
          "g_extreme" (a per-(head, channel) coin, then g = -U(8, 20) on the
          channels whose coin came up and -U(0.01, 0.5) on the others: every
          16-token chunk then spans a log-decay far beyond the fp32 range of
          e^{-G} on half of the channels), or "none".
    beta: "logits" (b ~ N(0,1)), "values" (beta ~ U(0,1)), both in the input dtype.
    h0_std: standard deviation of the fp32 initial state, or None for no h0.
    scale: output scale; defaults to K^-0.5.
    v_std: standard deviation of v (defaults to qkv_std).
    """
    gen = _gen(seed)
    cu_seqlens = None
    N = B
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        N = len(lengths)
        T = sum(lengths)
        B = 1
        cu = [0]
        for n in lengths:
            cu.append(cu[-1] + n)
        cu_seqlens = torch.tensor(cu, dtype=torch.int32)
    q = _randn(gen, (B, T, H, K), dtype, qkv_std)
    k = _randn(gen, (B, T, H, K), dtype, qkv_std)
    v = _randn(gen, (B, T, H, V), dtype, qkv_std if v_std is None else v_std)
    out = dict(q=q, k=k, v=v, g=None, g_head=None, a=None, dt_bias=None, A_log=None, beta=None, b=None,
               h0=None, cu_seqlens=cu_seqlens, N=N, B=B, T=T, H=H, K=K, V=V, dtype=dtype,
               gate=gate, beta_mode=beta, l2norm=l2norm, delta=delta,
               scale=(1.0 / math.sqrt(K)) if scale is None else float(scale))
    if gate == "inputs":
        out["a"] = _randn(gen, (B, T, H * K), torch.float32)
        out["dt_bias"] = _uniform(gen, (H * K,), -1.0, 1.0)
        out["A_log"] = _uniform(gen, (H,), 0.0, A_log_hi)
    elif gate == "g":
        out["g"] = -_uniform(gen, (B, T, H, K), 0.01, 3.0)
    elif gate == "head":
        out["g_head"] = -_uniform(gen, (B, T, H), 0.01, 3.0)
    elif gate == "g_extreme":
        fast = torch.rand(H, K, generator=gen) < 0.5
        hi = -_uniform(gen, (B, T, H, K), 8.0, 20.0)
        lo = -_uniform(gen, (B, T, H, K), 0.01, 0.5)
        out["g"] = torch.where(fast, hi, lo)
        out["gate"] = "g"
    elif gate != "none":
        raise ValueError(f"unknown gate mode {gate!r}")
    if beta == "logits":
        out["b"] = _randn(gen, (B, T, H), dtype)
    elif beta == "values":
        out["beta"] = _uniform(gen, (B, T, H), 0.0, 1.0, dtype)
    elif beta != "none":
        raise ValueError(f"unknown beta mode {beta!r}")
    if h0_std is not None:
        out["h0"] = _randn(gen, (N, H, V, K), torch.float32, h0_std)
    return out


def varlen_lengths(seed=3, n=16, lo=512, hi=8192):
    """Sequence lengths ~ U[lo, hi] (inclusive), drawn first from the seed."""
    gen = _gen(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def decode_workload(*, seed=4, B=256, H=32, HV=32, K=128, V=128, num_slots=512,
                    pad_frac=0.1, state_std=0.1, scale=None):
    """Inputs of one packed decode step.

    Draw order: packed qkv (bf16 [B, 2*H*K + HV*V] ~ N(0,1)), a (bf16 [B, HV*K]
    ~ N(0,1)), b (bf16 [B, HV] ~ N(0,1)), A_log (fp32 [HV] ~ U(0,2)), dt_bias
    (fp32 [HV*K] ~ U(-1,1)), state pool (fp32 [num_slots, HV, V, K] ~ state_std
    N(0,1)), slot indices (randperm(num_slots)[:B]), pad positions
    (randperm(B)[:round(pad_frac*B + 0.5)] set to -1).
    """
    gen = _gen(seed)
    packed = _randn(gen, (B, 2 * H * K + HV * V), torch.bfloat16)
    a = _randn(gen, (B, HV * K), torch.bfloat16)
    b = _randn(gen, (B, HV), torch.bfloat16)
    A_log = _uniform(gen, (HV,), 0.0, 2.0)
    dt_bias = _uniform(gen, (HV * K,), -1.0, 1.0)
    pool = _randn(gen, (num_slots, HV, V, K), torch.float32, state_std)
    if B > num_slots:
        raise ValueError("decode workload needs B <= num_slots (distinct slots)")
    idx = torch.randperm(num_slots, generator=gen)[:B].to(torch.int32)
    n_pad = int(math.floor(pad_frac * B + 0.5)) if pad_frac > 0 else 0
    if n_pad:
        pads = torch.randperm(B, generator=gen)[:n_pad]
        idx[pads] = -1
    return dict(packed_qkv=packed, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state_pool=pool,
                indices=idx, B=B, H=H, HV=HV, K=K, V=V, num_slots=num_slots,
                scale=(1.0 / math.sqrt(K)) if scale is None else float(scale))


def decode_conv_workload(*, seed=6, W=4, bias=True, **kw):
    """A decode workload (decode_workload with the same arguments, drawn first)
    plus the conv in front of it: conv state bf16 [num_slots, W-1, C] ~ N(0,1),
    conv weight fp32 [C, W] ~ N(0, 1/W), conv bias fp32 [C] ~ N(0, 0.1^2) (or
    None), C = 2*H*K + HV*V; the packed row is then the conv input."""
    out = decode_workload(seed=seed, **kw)
    gen = _gen(seed + 1000)
    C = out["packed_qkv"].shape[1]
    out["conv_state"] = _randn(gen, (out["num_slots"], W - 1, C), torch.bfloat16)
    out["conv_weight"] = _randn(gen, (C, W), torch.float32, 1.0 / math.sqrt(W))
    out["conv_bias"] = _randn(gen, (C,), torch.float32, 0.1) if bias else None
    out["W"] = W
    return out


def recurrent_workload(*, seed=5, B=64, T=8, H=32, HV=32, K=128, V=128, num_slots=128,
                       pad_frac=0.1, state_std=0.1, scale=None, A_log_range=(0.0, 2.0)):
    """Inputs of one short-T recurrent step (T tokens per row on a slot pool).

    Draw order: q, k (bf16 [B, T, H, K] ~ N(0,1)), v (bf16 [B, T, HV, V] ~ N(0,1)),
    a (bf16 [B, T, HV*K] ~ N(0,1)), b (bf16 [B, T, HV] ~ N(0,1)), A_log (fp32 [HV]
    ~ U(A_log_range), default U(0,2)), dt_bias (fp32 [HV*K] ~ U(-1,1)), state pool (fp32 [num_slots, HV,
    V, K] ~ state_std N(0,1)), slot indices (randperm(num_slots)[:B]), pad
    positions (randperm(B)[:round(pad_frac*B + 0.5)] set to -1).
    """
    gen = _gen(seed)
    q = _randn(gen, (B, T, H, K), torch.bfloat16)
    k = _randn(gen, (B, T, H, K), torch.bfloat16)
    v = _randn(gen, (B, T, HV, V), torch.bfloat16)
    a = _randn(gen, (B, T, HV * K), torch.bfloat16)
    b = _randn(gen, (B, T, HV), torch.bfloat16)
    A_log = _uniform(gen, (HV,), float(A_log_range[0]), float(A_log_range[1]))
    dt_bias = _uniform(gen, (HV * K,), -1.0, 1.0)
    pool = _randn(gen, (num_slots, HV, V, K), torch.float32, state_std)
    if B > num_slots:
        raise ValueError("recurrent workload needs B <= num_slots (distinct slots)")
    idx = torch.randperm(num_slots, generator=gen)[:B].to(torch.int32)
    n_pad = int(math.floor(pad_frac * B + 0.5)) if pad_frac > 0 else 0
    if n_pad:
        pads = torch.randperm(B, generator=gen)[:n_pad]
        idx[pads] = -1
    return dict(q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state_pool=pool, indices=idx,
                B=B, T=T, H=H, HV=HV, K=K, V=V, num_slots=num_slots,
                scale=(1.0 / math.sqrt(K)) if scale is None else float(scale))


# The five benchmark settings, by name.
def fp32_small(seed=0, **kw):
    return chunk_workload(seed=seed, B=1, T=128, H=2, K=64, V=64, dtype=torch.float32,
                          A_log_hi=1.0, h0_std=None, **kw)


def linear_attn(seed=1, **kw):
    kw.setdefault("T", 1024)
    return chunk_workload(seed=seed, B=2, H=4, K=128, V=128, dtype=torch.bfloat16, gate="none",
                          beta="none", l2norm=False, delta=False, h0_std=None,
                          qkv_std=1.0 / math.sqrt(128), scale=1.0, **kw)


def prefill(seed=2, **kw):
    kw.setdefault("T", 8192)
    kw.setdefault("H", 32)
    return chunk_workload(seed=seed, B=1, K=128, V=128, dtype=torch.bfloat16, **kw)


def varlen(seed=3, n=16, lo=512, hi=8192, **kw):
    kw.setdefault("H", 32)
    return chunk_workload(seed=seed, lengths=varlen_lengths(seed, n, lo, hi), K=128, V=128,
                          dtype=torch.bfloat16, **kw)


def decode(seed=4, **kw):
    return decode_workload(seed=seed, **kw)
