"""GPU parity of kda_decode_conv_step (the decode step with its causal conv1d +
SiLU in front) against the fp64 oracle through the C ABI: o and the updated
state slots within the bf16 tolerances, the conv state bit-exact (it only
moves bf16 inputs), padding rows and untouched slots bit-exact."""

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


def _run(wl, in_place):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in wl.items()}
    cn = Canary()
    pool = cn.clone(d["state_pool"], "state pool")
    cs_in = cn.clone(d["conv_state"], "conv state")
    cs_out = cs_in if in_place else cn.clone(cs_in, "conv state out")
    o = cn.empty((d["packed_qkv"].shape[0], wl["HV"], wl["V"]), torch.bfloat16, name="o")
    kda.kda_decode_conv_step(d["packed_qkv"], cs_in, d["conv_weight"], d["conv_bias"], d["a"], d["b"],
                             d["A_log"], d["dt_bias"], pool, d["indices"], H=wl["H"], HV=wl["HV"], K=wl["K"],
                             V=wl["V"], scale=wl["scale"], conv_state_out=cs_out, o=o)
    cn.check()
    return o, pool, cs_out


def _check(wl, in_place):
    o, pool, cs = _run(wl, in_place)
    o_ref, pool_ref, cs_ref = ko.kda_decode_conv(
        np64(wl["packed_qkv"]), np64(wl["conv_state"]), np64(wl["conv_weight"]), np64(wl["conv_bias"]),
        np64(wl["a"]), np64(wl["b"]), np64(wl["A_log"]), np64(wl["dt_bias"]), np64(wl["state_pool"]),
        wl["indices"].numpy(), H=wl["H"], HV=wl["HV"], K=wl["K"], V=wl["V"], scale=wl["scale"])
    idx = wl["indices"]
    valid = idx[idx >= 0].long()
    assert_close("decode+conv o", np64(o), o_ref, torch.bfloat16)
    assert_close("decode+conv state", np64(pool[valid.cuda()]), pool_ref[valid.numpy()], torch.bfloat16)
    # the conv state of the valid slots: shifted inputs, exact
    assert torch.equal(cs[valid.cuda()].float().cpu(), torch.from_numpy(cs_ref[valid.numpy()]).float())
    pads = (idx < 0).nonzero().flatten().cuda()
    assert torch.equal(o[pads], torch.zeros_like(o[pads]))
    untouched = torch.ones(wl["num_slots"], dtype=torch.bool)
    untouched[valid] = False
    ut = untouched.nonzero().flatten().cuda()
    assert torch.equal(pool[ut], wl["state_pool"].cuda()[ut])
    if in_place:
        assert torch.equal(cs[ut], wl["conv_state"].cuda()[ut])


@pytest.mark.parametrize("B,H,HV,K,V,Wd,bias,in_place", [
    (5, 2, 2, 128, 128, 4, True, True),    # in place (HV == H)
    (7, 1, 4, 64, 64, 3, False, False),    # HV = 4H: separate conv-state output, no bias
    (6, 2, 4, 128, 64, 2, True, False),
    (9, 2, 2, 64, 128, 4, True, False),
])
def test_decode_conv_small(B, H, HV, K, V, Wd, bias, in_place):
    wl = W.decode_conv_workload(seed=130 + B, W=Wd, bias=bias, B=B, H=H, HV=HV, K=K, V=V, num_slots=2 * B + 3,
                                pad_frac=0.25)
    _check(wl, in_place)


def test_decode_conv_full_size():
    """The decode benchmark setting (B=256, H=HV=32, K=V=128, 26 pads) with a width-4 conv, in place."""
    _check(W.decode_conv_workload(W=4), in_place=True)
