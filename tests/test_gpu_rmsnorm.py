"""GPU parity of kda_head_rmsnorm (output-side per-head RMSNorm) against the
fp64 oracle through the C ABI, on bf16 inputs: |y - y_ref| within bf16
rounding of y (rel <= 2^-7 elementwise plus a small absolute floor)."""

import numpy as np
import pytest
import torch

import kimi_delta_attention_04_gb300 as kda
from kimi_delta_attention_04_gb300 import workloads as W
from oracle import kda_oracle as ko

from kda_cases import Canary, gpu_chunk, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_04_gb300 import build
    build.build()
    kda.load()


def _check(y, x, w, eps):
    ref = ko.head_rmsnorm(np64(x), np64(w), eps)
    err = np.abs(np64(y) - ref)
    assert np.all(err <= 2.0 ** -7 * np.abs(ref) + 1e-6), float(err.max())


@pytest.mark.parametrize("V", [64, 128])
def test_rmsnorm_random_rows(V):
    gen = torch.Generator().manual_seed(120 + V)
    x = (torch.randn(37, 3, V, generator=gen) * torch.logspace(-3, 2, 37).view(37, 1, 1)).to(torch.bfloat16)
    x[5, 1] = 0  # an all-zero row stays zero
    w = torch.rand(V, generator=gen) * 2 - 0.5
    xd, wd = x.cuda(), w.cuda()
    cn = Canary()
    y = cn.empty(tuple(x.shape), torch.bfloat16, name="y")
    kda.kda_head_rmsnorm(xd, wd, eps=1e-6, out=y)
    cn.check()
    _check(y, x, w, 1e-6)
    assert torch.all(y[5, 1] == 0)
    kda.kda_head_rmsnorm(xd, wd, eps=1e-6, out=xd)  # in place
    torch.cuda.synchronize()
    assert torch.equal(xd, y)


def test_rmsnorm_on_chunk_forward_output():
    """The norm applied to a prefill's o (the place the pages put it)."""
    wl = W.prefill(T=300, H=4, seed=121)
    o, _ = gpu_chunk(wl)
    w = torch.linspace(0.5, 1.5, wl["V"])
    y = kda.kda_head_rmsnorm(o, w.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    _check(y, o.cpu(), w, 1e-5)
