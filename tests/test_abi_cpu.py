"""C-ABI checks that need no GPU: the library loads, exports what include/kda.h
declares, its structs match the ctypes mirrors byte for byte, and host-side
validation rejects bad arguments before anything is launched."""

import ctypes
import re
import subprocess
from pathlib import Path

import pytest

import kimi_delta_attention_04_gb300 as kda
from kimi_delta_attention_04_gb300 import _lib
from kimi_delta_attention_04_gb300 import build as kbuild

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "kda.h"


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return _lib.load()


def _declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert _declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(_lib.lib_path())], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared_functions():
        assert name in exported, f"{name} declared in kda.h but not exported"
        assert hasattr(lib, name)


def test_version_string(lib):
    assert kda.version().startswith("kda-gb300")


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    fields_c = [f for f, _ in _lib.ChunkArgs._fields_]
    fields_d = [f for f, _ in _lib.DecodeArgs._fields_]
    fields_r = [f for f, _ in _lib.RecurrentArgs._fields_]
    fields_n = [f for f, _ in _lib.RmsNormArgs._fields_]
    fields_c2 = [f for f, _ in _lib.DecodeConvArgs._fields_]
    fields_p = [f for f, _ in _lib.Tcgen05ProbeArgs._fields_]
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void){"]
    lines.append('printf("chunk %zu\\n", sizeof(kda_chunk_args));')
    for f in fields_c:
        lines.append(f'printf("c.{f} %zu\\n", offsetof(kda_chunk_args, {f}));')
    lines.append('printf("decode %zu\\n", sizeof(kda_decode_args));')
    for f in fields_d:
        lines.append(f'printf("d.{f} %zu\\n", offsetof(kda_decode_args, {f}));')
    lines.append('printf("recurrent %zu\\n", sizeof(kda_recurrent_args));')
    for f in fields_r:
        lines.append(f'printf("r.{f} %zu\\n", offsetof(kda_recurrent_args, {f}));')
    lines.append('printf("maxT %d\\n", KDA_RECURRENT_MAX_T);')
    lines.append('printf("rmsnorm %zu\\n", sizeof(kda_rmsnorm_args));')
    lines.append('printf("dconv %zu\\n", sizeof(kda_decode_conv_args));')
    for f in fields_c2:
        lines.append(f'printf("dc.{f} %zu\\n", offsetof(kda_decode_conv_args, {f}));')
    for f in fields_n:
        lines.append(f'printf("n.{f} %zu\\n", offsetof(kda_rmsnorm_args, {f}));')
    lines.append('printf("probe %zu\\n", sizeof(kda_tcgen05_probe_args));')
    for f in fields_p:
        lines.append(f'printf("p.{f} %zu\\n", offsetof(kda_tcgen05_probe_args, {f}));')
    lines.append("return 0;}")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(got["chunk"]) == ctypes.sizeof(_lib.ChunkArgs)
    assert int(got["decode"]) == ctypes.sizeof(_lib.DecodeArgs)
    for f in fields_c:
        assert int(got[f"c.{f}"]) == getattr(_lib.ChunkArgs, f).offset, f
    for f in fields_d:
        assert int(got[f"d.{f}"]) == getattr(_lib.DecodeArgs, f).offset, f
    assert int(got["recurrent"]) == ctypes.sizeof(_lib.RecurrentArgs)
    for f in fields_r:
        assert int(got[f"r.{f}"]) == getattr(_lib.RecurrentArgs, f).offset, f
    assert int(got["maxT"]) == _lib.KDA_RECURRENT_MAX_T
    assert int(got["rmsnorm"]) == ctypes.sizeof(_lib.RmsNormArgs)
    assert int(got["dconv"]) == ctypes.sizeof(_lib.DecodeConvArgs)
    for f in fields_c2:
        assert int(got[f"dc.{f}"]) == getattr(_lib.DecodeConvArgs, f).offset, f
    for f in fields_n:
        assert int(got[f"n.{f}"]) == getattr(_lib.RmsNormArgs, f).offset, f
    assert int(got["probe"]) == ctypes.sizeof(_lib.Tcgen05ProbeArgs)
    for f in fields_p:
        assert int(got[f"p.{f}"]) == getattr(_lib.Tcgen05ProbeArgs, f).offset, f


# --- host-side validation, exercised with fake (never dereferenced) pointers ---

FAKE = 0x10000  # 64 KiB: aligned to anything the library checks


def _chunk(**over):
    a = _lib.ChunkArgs()
    a.dtype, a.B, a.T, a.H, a.dk, a.dv, a.N = _lib.KDA_DTYPE_BF16, 1, 100, 2, 128, 128, 1
    a.gate_mode, a.beta_mode, a.flags, a.scale = _lib.KDA_GATE_G, _lib.KDA_BETA_LOGITS, _lib.KDA_FLAG_L2NORM_QK, 0.1
    a.q = a.k = a.v = a.g = a.beta = a.o = FAKE
    for k, v in over.items():
        setattr(a, k, v)
    return a


def _ws(lib, a):
    return int(lib.kda_chunk_workspace_size(ctypes.byref(a)))


def _fwd(lib, a, ws_ptr=FAKE, ws_bytes=1 << 40):
    return lib.kda_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes), None)


def test_workspace_size_formula(lib):
    a = _chunk()
    # bf16 d=128 runs the fused kernel: the varlen plan header (N + 2 int32, rounded to 256),
    # then a fixed pool: a 256-byte map of 40 per-cluster rings, each 16 slots of one
    # prepared chunk (3 x 128 x 16 16-bit operands, 16 x 24 Mqk, 128 gamma, 16 output
    # factors, 128 x 16 U~)
    slot = 3 * 128 * 16 * 2 + 16 * 24 * 2 + 128 * 4 + 16 * 4 + 128 * 16 * 4
    pool = 256 + 40 * 16 * slot
    assert _ws(lib, a) == 256 + pool
    assert _ws(lib, _chunk(cu_seqlens=FAKE, N=100)) == 512 + pool
    assert _ws(lib, a) <= _lib.KDA_NOALLOC_SCRATCH_BYTES  # the no-alloc entry point covers this path
    # two-kernel path: header + ceil(100/16) chunks * H * record
    a.dk = a.dv = 64
    rec64 = 3 * 16 * 64 * 2 + 64 * 16 * 4 + 16 * 16 * 2 + 64 * 4
    assert _ws(lib, a) == 256 + 7 * 2 * rec64
    # varlen: one extra partial chunk per sequence at most
    v = _chunk(cu_seqlens=FAKE, N=4, dk=64, dv=64)
    assert _ws(lib, v) == 256 + (7 + 4) * 2 * rec64
    f = _chunk(dtype=_lib.KDA_DTYPE_FP32, dk=64, dv=128)
    recf = 3 * 16 * 64 * 4 + 128 * 16 * 4 + 16 * 16 * 4 + 64 * 4
    assert _ws(lib, f) == 256 + 7 * 2 * recf
    # per-chunk states and the output pass run on the same fused kernel: same pool
    assert _ws(lib, _chunk(h_chunks=FAKE)) == 256 + pool
    assert _ws(lib, _chunk(h_chunks=FAKE, T=100000)) == 256 + pool


@pytest.mark.parametrize("over,status", [
    (dict(q=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(o=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), _lib.KDA_ERR_INVALID_ARG),              # misaligned
    (dict(g=None), _lib.KDA_ERR_INVALID_ARG),                  # GATE_G without g
    (dict(beta=None), _lib.KDA_ERR_INVALID_ARG),               # delta rule without beta
    (dict(gate_mode=7), _lib.KDA_ERR_INVALID_ARG),
    (dict(beta_mode=5), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=0x80), _lib.KDA_ERR_INVALID_ARG),
    (dict(dtype=9), _lib.KDA_ERR_INVALID_ARG),
    (dict(H=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(T=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(N=2), _lib.KDA_ERR_INVALID_ARG),                     # N != B without cu_seqlens
    (dict(B=2, N=2, cu_seqlens=FAKE), _lib.KDA_ERR_INVALID_ARG),  # varlen needs B == 1
    (dict(dk=96, dv=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dk=64, dv=128), _lib.KDA_ERR_UNSUPPORTED),           # bf16 path needs dk == dv
    (dict(gate_mode=_lib.KDA_GATE_INPUTS, a=FAKE, A_log=None, dt_bias=FAKE), _lib.KDA_ERR_INVALID_ARG),
    (dict(h0=FAKE + 8), _lib.KDA_ERR_INVALID_ARG),
    (dict(h_chunks=FAKE + 8), _lib.KDA_ERR_INVALID_ARG),       # per-chunk states need 16-byte alignment
    (dict(h_chunks=FAKE, dtype=_lib.KDA_DTYPE_FP32, dk=64, dv=64), _lib.KDA_ERR_UNSUPPORTED),  # bf16 only
])
def test_chunk_validation_rejects(lib, over, status):
    a = _chunk(**over)
    assert _ws(lib, a) == 0
    assert _fwd(lib, a) == status
    assert lib.kda_chunk_output(ctypes.byref(a), ctypes.c_void_p(FAKE), ctypes.c_size_t(1 << 40), None) == status


def test_selftest_bounded_wait_validation(lib):
    """The wait self-test needs an aligned status word and a limit in [1 us, 10 s]."""
    f = lib.kda_selftest_bounded_wait
    assert f(None, 1_000_000, None) == _lib.KDA_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(FAKE + 2), 1_000_000, None) == _lib.KDA_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(FAKE), 999, None) == _lib.KDA_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(FAKE), 10_000_000_001, None) == _lib.KDA_ERR_INVALID_ARG


def _probe(**over):
    a = _lib.Tcgen05ProbeArgs()
    a.K, a.N, a.layout, a.a_from_tmem, a.reps = 16, 64, 0, 0, 10
    a.a = a.b = a.d = a.cycles = a.err = FAKE
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over", [dict(K=8), dict(K=48), dict(K=256), dict(N=8), dict(N=24), dict(N=272),
                                  dict(layout=2), dict(a_from_tmem=2), dict(reps=-1), dict(reps=4097),
                                  dict(a=None), dict(b=None), dict(d=None), dict(a=FAKE + 8), dict(d=FAKE + 4),
                                  dict(cycles=FAKE + 4), dict(err=FAKE + 2)])
def test_selftest_tcgen05_validation(lib, over):
    """The tcgen05 probe checks its shape, layout and pointers before launching."""
    a = _probe(**over)
    assert lib.kda_selftest_tcgen05(ctypes.byref(a), None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_selftest_tcgen05(None, None) == _lib.KDA_ERR_INVALID_ARG


def test_chunk_output_needs_states(lib):
    """The chunk-parallel output pass reads h_chunks: without it the call is refused."""
    a = _chunk()
    assert lib.kda_chunk_output(ctypes.byref(a), ctypes.c_void_p(FAKE), ctypes.c_size_t(1 << 40), None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_output(None, None, 0, None) == _lib.KDA_ERR_INVALID_ARG


def test_chunk_workspace_checks(lib):
    a = _chunk()
    need = _ws(lib, a)
    assert _fwd(lib, a, ws_ptr=0) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, a, ws_bytes=need - 1) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, a, ws_ptr=FAKE + 16) == _lib.KDA_ERR_INVALID_ARG  # needs 256-byte alignment
    assert lib.kda_chunk_fwd(None, None, 0, None) == _lib.KDA_ERR_INVALID_ARG


def _dec(**over):
    a = _lib.DecodeArgs()
    a.B, a.H, a.HV, a.K, a.V, a.num_slots, a.flags, a.scale = 4, 2, 4, 128, 128, 8, _lib.KDA_FLAG_L2NORM_QK, 0.1
    a.packed_qkv = a.a = a.b = a.A_log = a.dt_bias = a.state_pool = a.indices = a.o = FAKE
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,status", [
    (dict(HV=3), _lib.KDA_ERR_INVALID_ARG),                   # HV not a multiple of H
    (dict(K=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(V=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(indices=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(state_pool=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(packed_qkv=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=0x2), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=0x8), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=_lib.KDA_FLAG_CHECK_INDICES), _lib.KDA_ERR_INVALID_ARG),  # the debug check needs err
    (dict(B=-1), _lib.KDA_ERR_INVALID_ARG),
])
def test_decode_validation_rejects(lib, over, status):
    a = _dec(**over)
    assert lib.kda_decode_step(ctypes.byref(a), None) == status


def _rec(**over):
    a = _lib.RecurrentArgs()
    a.B, a.T, a.H, a.HV, a.K, a.V, a.num_slots = 4, 8, 2, 4, 128, 128, 8
    a.flags, a.scale = _lib.KDA_FLAG_L2NORM_QK, 0.1
    a.q = a.k = a.v = a.a = a.b = a.A_log = a.dt_bias = a.state_pool = a.indices = a.o = FAKE
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,status", [
    (dict(HV=3), _lib.KDA_ERR_INVALID_ARG),                   # HV not a multiple of H
    (dict(T=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(T=_lib.KDA_RECURRENT_MAX_T + 1), _lib.KDA_ERR_UNSUPPORTED),  # long sequences: chunk forward
    (dict(K=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(V=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(q=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(indices=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(state_pool=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(v=FAKE + 4), _lib.KDA_ERR_INVALID_ARG),              # misaligned
    (dict(flags=0x2), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=_lib.KDA_FLAG_CHECK_INDICES), _lib.KDA_ERR_INVALID_ARG),  # the debug check needs err
    (dict(B=-1), _lib.KDA_ERR_INVALID_ARG),
])
def test_recurrent_validation_rejects(lib, over, status):
    a = _rec(**over)
    assert lib.kda_recurrent_step(ctypes.byref(a), None) == status
    assert lib.kda_recurrent_step(None, None) == _lib.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("over,status", [
    (dict(W=1), _lib.KDA_ERR_UNSUPPORTED),
    (dict(W=5), _lib.KDA_ERR_UNSUPPORTED),
    (dict(conv_state_in=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(conv_weight=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(conv_state_out=FAKE), _lib.KDA_ERR_INVALID_ARG),       # in place with HV = 2H races
    (dict(conv_bias=FAKE + 2), _lib.KDA_ERR_INVALID_ARG),        # misaligned
])
def test_decode_conv_validation_rejects(lib, over, status):
    a = _lib.DecodeConvArgs()
    a.dec = _dec()                  # H = 2, HV = 4
    a.W, a.conv_state_in, a.conv_state_out, a.conv_weight, a.conv_bias = 4, FAKE, FAKE + 0x1000, FAKE, None
    for k, v in over.items():
        setattr(a, k, v)
    assert lib.kda_decode_conv_step(ctypes.byref(a), None) == status


@pytest.mark.parametrize("over,status", [
    (dict(V=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(R=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(x=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(weight=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(y=FAKE + 2), _lib.KDA_ERR_INVALID_ARG),   # misaligned
    (dict(eps=-1.0), _lib.KDA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), _lib.KDA_ERR_INVALID_ARG),
])
def test_rmsnorm_validation_rejects(lib, over, status):
    a = _lib.RmsNormArgs()
    a.R, a.V, a.eps = 10, 128, 1e-6
    a.x = a.weight = a.y = FAKE
    for k, v in over.items():
        setattr(a, k, v)
    assert lib.kda_head_rmsnorm(ctypes.byref(a), None) == status


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 16, 1, 64)
    with pytest.raises((ValueError, RuntimeError)):
        kda.kda_chunk_fwd(q, q, q, scale=1.0, delta=False)
