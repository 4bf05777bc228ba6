"""GPU parity of kda_recurrent_step (T tokens per row on a state-slot pool)
against the fp64 oracle, through the C ABI (ctypes binding) on the same
bf16-rounded inputs. Below 8 tokens the call runs the per-token kernel, from
8 the chunk-form kernel; the cases cover both sides of the switch. Tolerances as for decode: rel-Frobenius <= 5e-3 and
max-abs <= 2e-2 for o and the updated slots; padding rows and slots no row
indexes are bit-exact."""

import pytest
import torch

import kimi_delta_attention_04_gb300 as kda
from kimi_delta_attention_04_gb300 import workloads as W
from oracle import kda_oracle as ko

from kda_cases import Canary, assert_close, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_04_gb300 import build
    build.build()
    kda.load()


def _run(wl, err=None):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in wl.items()}
    cn = Canary()
    pool = cn.clone(d["state_pool"], "state pool")
    o = cn.empty((d["q"].shape[0], d["q"].shape[1], d["v"].shape[2], d["v"].shape[3]), torch.bfloat16, name="o")
    kda.kda_recurrent_step(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], pool, d["indices"],
                           scale=wl["scale"], err=err, l2norm_qk=wl.get("l2norm", True), o=o)
    cn.check()
    return o, pool


def _oracle(wl):
    return ko.kda_recurrent_pool(np64(wl["q"]), np64(wl["k"]), np64(wl["v"]), np64(wl["a"]), np64(wl["b"]),
                                 np64(wl["A_log"]), np64(wl["dt_bias"]), np64(wl["state_pool"]),
                                 wl["indices"].numpy(), scale=wl["scale"], l2norm_qk=wl.get("l2norm", True))


def _check(wl):
    o, pool = _run(wl)
    o_ref, pool_ref = _oracle(wl)
    idx = wl["indices"]
    valid = idx[idx >= 0].long()
    assert_close("recurrent o", np64(o), o_ref, torch.bfloat16)
    assert_close("recurrent state", np64(pool[valid.cuda()]), pool_ref[valid.numpy()], torch.bfloat16)
    pads = (idx < 0).nonzero().flatten().cuda()
    assert torch.equal(o[pads], torch.zeros_like(o[pads]))
    untouched = torch.ones(wl["num_slots"], dtype=torch.bool)
    untouched[valid] = False
    ut = untouched.nonzero().flatten().cuda()
    assert torch.equal(pool[ut], wl["state_pool"].cuda()[ut])
    return o, pool


@pytest.mark.parametrize("B,T,H,HV,K,V", [
    (4, 3, 2, 4, 64, 64),      # value-head grouping, ragged T
    (5, 8, 2, 2, 128, 128),
    (3, 33, 1, 2, 128, 64),    # more tokens than one warp's share, HV = 2H
    (6, 1, 2, 4, 64, 128),     # T = 1
    (2, 64, 1, 1, 128, 128),   # the longest T the entry point takes
    (5, 7, 2, 4, 128, 128),    # the per-token kernel's longest T
    (5, 16, 2, 2, 128, 128),   # the chunk kernel on one full chunk
    (3, 17, 2, 4, 64, 128),    # two chunks, the second of one token
])
def test_recurrent_small(B, T, H, HV, K, V):
    wl = W.recurrent_workload(seed=90 + B + T, B=B, T=T, H=H, HV=HV, K=K, V=V, num_slots=2 * B + 3, pad_frac=0.25)
    _check(wl)


@pytest.mark.parametrize("T", [5, 16, 40])
def test_recurrent_extreme_gates(T):
    """A_log ~ U(2.5, 3): log-decays of about -2 to -80 per token, so a 16-token
    chunk spans far more than the -88 at which e^{-G} overflows fp32; both the
    per-token kernel (T < 8) and the chunk-form kernel (T >= 8) must stay finite
    and meet the bf16 tolerance."""
    wl = W.recurrent_workload(seed=190 + T, B=6, T=T, H=2, HV=4, num_slots=9, A_log_range=(2.5, 3.0))
    o, pool = _check(wl)
    assert torch.isfinite(o.float()).all() and torch.isfinite(pool).all()


def test_recurrent_full_size():
    """B=64 rows of T=8 tokens, H=HV=32, K=V=128, fp32 pool [128, 32, 128, 128], 6 padded rows."""
    _check(W.recurrent_workload())


def test_recurrent_full_size_long():
    """B=64 rows of T=64 tokens (four chunks each), H=HV=32, K=V=128, fp32 pool
    [128, 32, 128, 128], 6 padded rows: the long recurrent step of the benchmark.
    Each CTA keeps its state in tensor memory between chunks, and there are more
    CTAs than fit on the GPU at once, so later ones allocate columns that earlier
    ones released; every valid row is compared with the oracle."""
    _check(W.recurrent_workload(seed=5, B=64, T=64, num_slots=128))


def test_recurrent_t1_matches_decode_kernel():
    """One token per row through both entry points (decode reads a packed row)."""
    wl = W.recurrent_workload(seed=97, B=9, T=1, H=2, HV=4, K=128, V=128, num_slots=12, pad_frac=0.2)
    o, pool = _run(wl)
    B, H, HV, K, V = wl["B"], wl["H"], wl["HV"], wl["K"], wl["V"]
    packed = torch.cat([wl["q"].reshape(B, H * K), wl["k"].reshape(B, H * K), wl["v"].reshape(B, HV * V)], dim=1)
    pool2 = wl["state_pool"].cuda().clone()
    o2 = kda.kda_decode_step(packed.cuda().contiguous(), wl["a"].reshape(B, HV * K).cuda().contiguous(),
                             wl["b"].reshape(B, HV).cuda().contiguous(), wl["A_log"].cuda(), wl["dt_bias"].cuda(),
                             pool2, wl["indices"].cuda(), H=H, HV=HV, K=K, V=V, scale=wl["scale"])
    torch.cuda.synchronize()
    assert_close("o vs decode", np64(o[:, 0]), np64(o2), torch.bfloat16)
    assert_close("state vs decode", np64(pool), np64(pool2), torch.bfloat16)


def test_recurrent_bad_slot_and_padding():
    wl = W.recurrent_workload(seed=98, B=5, T=4, H=2, HV=2, K=64, V=64, num_slots=6, pad_frac=0.0)
    wl["indices"] = torch.tensor([-1, 4, 77, 0, -1], dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, pool = _run(wl, err=err)
    assert int(err.item()) == 1  # KDA_ERR_INVALID_ARG from the out-of-range slot
    assert torch.equal(o[[0, 2, 4]], torch.zeros_like(o[[0, 2, 4]]))
    assert torch.equal(pool[[1, 2, 3, 5]], wl["state_pool"].cuda()[[1, 2, 3, 5]])
    o_ref, pool_ref = _oracle(dict(wl, indices=torch.tensor([-1, 4, -1, 0, -1], dtype=torch.int32)))
    assert_close("recurrent o", np64(o), o_ref, torch.bfloat16)
    assert_close("recurrent state", np64(pool[[0, 4]]), pool_ref[[0, 4]], torch.bfloat16)


def test_recurrent_split_tokens_equals_one_call():
    """T tokens in one call equal T1 then T - T1 tokens in two calls on the same pool."""
    wl = W.recurrent_workload(seed=99, B=4, T=10, H=2, HV=4, K=128, V=128, num_slots=8, pad_frac=0.25)
    o, pool = _run(wl)
    first = {k: (v[:, :6].contiguous() if k in ("q", "k", "v", "a", "b") else v) for k, v in wl.items()}
    o1, pool1 = _run(first)
    second = {k: (v[:, 6:].contiguous() if k in ("q", "k", "v", "a", "b") else v) for k, v in wl.items()}
    second["state_pool"] = pool1.cpu()
    o2, pool2 = _run(second)
    assert_close("o split", np64(torch.cat([o1, o2], dim=1)), np64(o), torch.bfloat16)
    assert_close("state split", np64(pool2), np64(pool), torch.bfloat16)


@pytest.mark.parametrize("entry", ["decode", "recurrent"])
def test_check_indices_flag(entry):
    """KDA_FLAG_CHECK_INDICES: a repeated valid slot index is reported through err;
    distinct indices (pads and repeated -1s included) leave err at 0 and the
    results as without the check."""
    wl = W.recurrent_workload(seed=123, B=300, T=8, H=2, HV=2, K=64, V=64, num_slots=400, pad_frac=0.2)
    B, H, HV, K, V = wl["B"], wl["H"], wl["HV"], wl["K"], wl["V"]

    def call(indices, check):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pool = wl["state_pool"].cuda().clone()
        if entry == "recurrent":
            d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in wl.items()}
            o = kda.kda_recurrent_step(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], pool,
                                       indices.cuda(), scale=wl["scale"], err=err, check_indices=check)
        else:
            packed = torch.cat([wl["q"][:, 0].reshape(B, H * K), wl["k"][:, 0].reshape(B, H * K),
                                wl["v"][:, 0].reshape(B, HV * V)], dim=1).cuda().contiguous()
            o = kda.kda_decode_step(packed, wl["a"][:, 0].reshape(B, HV * K).cuda().contiguous(),
                                    wl["b"][:, 0].reshape(B, HV).cuda().contiguous(), wl["A_log"].cuda(),
                                    wl["dt_bias"].cuda(), pool, indices.cuda(), H=H, HV=HV, K=K, V=V,
                                    scale=wl["scale"], err=err, check_indices=check)
        torch.cuda.synchronize()
        return int(err.item()), o, pool

    idx = wl["indices"]
    assert int((idx < 0).sum()) > 1  # several pads share -1, which is not a repeat
    e0, o0, p0 = call(idx, False)
    e1, o1, p1 = call(idx, True)
    assert e0 == 0 and e1 == 0
    assert torch.equal(o0, o1) and torch.equal(p0, p1)
    dup = idx.clone()
    valid = (dup >= 0).nonzero().flatten()
    dup[valid[-1]] = dup[valid[3]]  # rows far apart (different check tiles) share a slot
    e2, _, _ = call(dup, True)
    assert e2 == 1


@pytest.mark.parametrize("T", [4, 12, 40])
def test_recurrent_without_l2norm(T):
    """KDA_FLAG_L2NORM_QK off (q, k used as given, drawn with std K^-1/2): the
    per-token kernel (T = 4) and the chunk-form kernel (T = 12, 40; bf16 level
    operands) against the oracle."""
    wl = W.recurrent_workload(seed=160 + T, B=6, T=T, H=2, HV=4, K=128, V=64, num_slots=9, pad_frac=0.2)
    s = 128 ** -0.5
    wl["q"] = (wl["q"].float() * s).to(torch.bfloat16)
    wl["k"] = (wl["k"].float() * s).to(torch.bfloat16)
    wl["l2norm"] = False
    _check(wl)


def test_decode_without_l2norm():
    """The packed decode with KDA_FLAG_L2NORM_QK off against the oracle's decode."""
    wl = W.decode_workload(seed=171, B=12, H=2, HV=4, K=64, V=128, num_slots=20, pad_frac=0.2)
    B, H, HV, K, V = wl["B"], wl["H"], wl["HV"], wl["K"], wl["V"]
    packed = wl["packed_qkv"].float()
    packed[:, : 2 * H * K] *= K ** -0.5
    packed = packed.to(torch.bfloat16)
    pool = wl["state_pool"].cuda().clone()
    o = kda.kda_decode_step(packed.cuda(), wl["a"].cuda(), wl["b"].cuda(), wl["A_log"].cuda(), wl["dt_bias"].cuda(),
                            pool, wl["indices"].cuda(), H=H, HV=HV, K=K, V=V, scale=wl["scale"], l2norm_qk=False)
    torch.cuda.synchronize()
    o_ref, pool_ref = ko.kda_decode(np64(packed), np64(wl["a"]), np64(wl["b"]), np64(wl["A_log"]),
                                    np64(wl["dt_bias"]), np64(wl["state_pool"]), wl["indices"].numpy(), H=H, HV=HV,
                                    K=K, V=V, scale=wl["scale"], l2norm_qk=False)
    valid = (wl["indices"] >= 0).nonzero().flatten()
    slots = wl["indices"][valid].long()
    assert_close("decode o (no l2norm)", np64(o)[valid.numpy()], o_ref[valid.numpy()], torch.bfloat16)
    assert_close("decode state (no l2norm)", np64(pool[slots.cuda()]), pool_ref[slots.numpy()], torch.bfloat16)
