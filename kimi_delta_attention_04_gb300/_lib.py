"""ctypes binding of libkda.so (include/kda.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. PyTorch supplies device memory, the current stream and the output
allocations. There is no CPU or PyTorch fallback: if libkda.so is missing or a
tensor is not on a CUDA device, the call raises.
"""

from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libkda.so"
_lock = threading.Lock()
_lib = None

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_TIMEOUT = 4
KDA_ERR_TOO_LARGE = 5
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
                4: "KDA_ERR_TIMEOUT", 5: "KDA_ERR_TOO_LARGE"}
KDA_NOALLOC_SCRATCH_BYTES = 16 << 20

KDA_DTYPE_BF16 = 0
KDA_DTYPE_FP32 = 1
KDA_GATE_NONE, KDA_GATE_G, KDA_GATE_INPUTS, KDA_GATE_HEAD_G = 0, 1, 2, 3
KDA_BETA_VALUES, KDA_BETA_LOGITS = 0, 1
KDA_FLAG_L2NORM_QK = 0x1
KDA_FLAG_DELTA_OFF = 0x2
KDA_FLAG_CHECK_INDICES = 0x4


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class ChunkArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32), ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("N", ctypes.c_int32),
        ("gate_mode", ctypes.c_int32), ("beta_mode", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("scale", ctypes.c_float),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("hT", ctypes.c_void_p), ("err", ctypes.c_void_p),
        ("h_chunks", ctypes.c_void_p),
    ]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("HV", ctypes.c_int32), ("K", ctypes.c_int32),
        ("V", ctypes.c_int32), ("num_slots", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("scale", ctypes.c_float),
        ("packed_qkv", ctypes.c_void_p), ("a", ctypes.c_void_p), ("b", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("state_pool", ctypes.c_void_p),
        ("indices", ctypes.c_void_p), ("o", ctypes.c_void_p), ("err", ctypes.c_void_p),
    ]


class DecodeConvArgs(ctypes.Structure):
    _fields_ = [
        ("dec", DecodeArgs), ("W", ctypes.c_int32), ("conv_state_in", ctypes.c_void_p),
        ("conv_state_out", ctypes.c_void_p), ("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
    ]


class RecurrentArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("HV", ctypes.c_int32),
        ("K", ctypes.c_int32), ("V", ctypes.c_int32), ("num_slots", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("scale", ctypes.c_float),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("a", ctypes.c_void_p),
        ("b", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("state_pool", ctypes.c_void_p), ("indices", ctypes.c_void_p), ("o", ctypes.c_void_p),
        ("err", ctypes.c_void_p),
    ]


KDA_RECURRENT_MAX_T = 64


class RmsNormArgs(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int64), ("V", ctypes.c_int32), ("eps", ctypes.c_float),
        ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("y", ctypes.c_void_p),
    ]


class Tcgen05ProbeArgs(ctypes.Structure):
    _fields_ = [
        ("K", ctypes.c_int32), ("N", ctypes.c_int32), ("layout", ctypes.c_int32), ("a_from_tmem", ctypes.c_int32),
        ("reps", ctypes.c_int32), ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("d", ctypes.c_void_p),
        ("cycles", ctypes.c_void_p), ("err", ctypes.c_void_p),
    ]


EXPORTS = ("kda_chunk_fwd", "kda_chunk_output", "kda_chunk_fwd_noalloc", "kda_chunk_workspace_size", "kda_decode_step",
           "kda_decode_conv_step", "kda_recurrent_step", "kda_head_rmsnorm", "kda_version",
           "kda_selftest_bounded_wait", "kda_selftest_tcgen05")


def lib_path() -> Path:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libkda.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _LIB_PATH.exists():
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -m kimi_delta_attention_04_gb300.build). There is no fallback path.")
        lib = ctypes.CDLL(str(_LIB_PATH))
        lib.kda_chunk_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd.argtypes = [ctypes.POINTER(ChunkArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.kda_chunk_output.restype = ctypes.c_int
        lib.kda_chunk_output.argtypes = [ctypes.POINTER(ChunkArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.kda_chunk_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_workspace_size.argtypes = [ctypes.POINTER(ChunkArgs)]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.c_void_p]
        lib.kda_recurrent_step.restype = ctypes.c_int
        lib.kda_recurrent_step.argtypes = [ctypes.POINTER(RecurrentArgs), ctypes.c_void_p]
        lib.kda_decode_conv_step.restype = ctypes.c_int
        lib.kda_decode_conv_step.argtypes = [ctypes.POINTER(DecodeConvArgs), ctypes.c_void_p]
        lib.kda_head_rmsnorm.restype = ctypes.c_int
        lib.kda_head_rmsnorm.argtypes = [ctypes.POINTER(RmsNormArgs), ctypes.c_void_p]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(ChunkArgs), ctypes.c_void_p]
        lib.kda_version.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        lib.kda_selftest_bounded_wait.restype = ctypes.c_int
        lib.kda_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
        lib.kda_selftest_tcgen05.restype = ctypes.c_int
        lib.kda_selftest_tcgen05.argtypes = [ctypes.POINTER(Tcgen05ProbeArgs), ctypes.c_void_p]
        _lib = lib
        return lib


def version() -> str:
    return load().kda_version().decode()


def selftest_bounded_wait(err, limit_ns, stream=None):
    """Run the bounded-wait self-test kernel: it waits on an mbarrier that nothing
    arrives on, gives up after limit_ns and writes KDA_ERR_TIMEOUT to err
    (a device int32 tensor). See include/kda.h."""
    with _on_device(err):
        st = load().kda_selftest_bounded_wait(_ptr(err), ctypes.c_uint64(int(limit_ns)), _stream_ptr(stream, err.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_bounded_wait")


def selftest_tcgen05(a, b, *, layout=0, a_from_tmem=False, reps=0, err=None, stream=None):
    """One tcgen05 MMA, d [128, N] = a [128, K] @ b[N, K]^T (bf16 in, fp32 out),
    and its timed round trips (see include/kda.h). Returns (d, cycles) with
    cycles an int64 CUDA tensor [7]: summed issue->done and issue->data cycles
    over `reps` round trips, the cycles of a burst of `reps` back-to-back
    groups on one accumulator, reps, the cycles of a burst over independent
    accumulators and their count, and the issuing thread's own cycles for the
    first burst."""
    K, N = int(a.shape[1]), int(b.shape[0])
    if a.shape[0] != 128 or b.shape[1] != K or a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise ValueError("expects bf16 a [128, K] and b [N, K]")
    d = torch.empty(128, N, dtype=torch.float32, device=a.device)
    cycles = torch.zeros(7, dtype=torch.int64, device=a.device)
    args = Tcgen05ProbeArgs()
    args.K, args.N, args.layout, args.a_from_tmem, args.reps = K, N, int(layout), int(bool(a_from_tmem)), int(reps)
    args.a, args.b, args.d, args.cycles, args.err = _ptr(a), _ptr(b), _ptr(d), _ptr(cycles), _ptr(err)
    with _on_device(a):
        st = load().kda_selftest_tcgen05(ctypes.byref(args), _stream_ptr(stream, a.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_tcgen05")
    return d, cycles


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t).__name__}")
    if not t.is_cuda:
        raise ValueError("libkda works on CUDA tensors only (no CPU fallback)")
    if not t.is_contiguous():
        raise ValueError("libkda needs contiguous tensors")
    return t.data_ptr()


def _stream_ptr(stream, device=None):
    """The stream to enqueue on: the given one, else the current stream of
    `device` (the device of the call's tensors)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _on_device(t):
    """Context in which a C call runs: the device of tensor t is made current,
    so the library's per-device state (kernel attributes, the no-allocation
    scratch address) and its launches refer to the device that holds the data."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("libkda works on CUDA tensors only (no CPU fallback)")
    return torch.cuda.device(t.device)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return KDA_DTYPE_BF16
    if dt == torch.float32:
        return KDA_DTYPE_FP32
    raise ValueError(f"unsupported input dtype {dt}; use torch.bfloat16 or torch.float32")


def make_chunk_args(q, k, v, *, scale, g=None, a=None, dt_bias=None, A_log=None, beta=None, b=None,
                    h0=None, cu_seqlens=None, l2norm_qk=False, delta=True, o=None, hT=None, err=None, g_head=None,
                    h_chunks=None):
    """Fill the C argument struct from tensors (no allocation, no launch)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if g is not None:
        gate_mode = KDA_GATE_G
    elif g_head is not None:
        gate_mode, g = KDA_GATE_HEAD_G, g_head  # passed in the g field
    elif a is not None:
        gate_mode = KDA_GATE_INPUTS
    else:
        gate_mode = KDA_GATE_NONE
    if beta is not None:
        beta_mode, beta_t = KDA_BETA_VALUES, beta
    else:
        beta_mode, beta_t = KDA_BETA_LOGITS, b
    flags = (KDA_FLAG_L2NORM_QK if l2norm_qk else 0) | (0 if delta else KDA_FLAG_DELTA_OFF)
    args = ChunkArgs()
    args.dtype = _dtype_code(q.dtype)
    args.B, args.T, args.H, args.dk, args.dv, args.N = B, T, H, dk, dv, N
    args.gate_mode, args.beta_mode, args.flags = gate_mode, beta_mode, flags
    args.scale = float(scale)
    args.q, args.k, args.v = _ptr(q), _ptr(k), _ptr(v)
    args.g, args.a, args.A_log, args.dt_bias = _ptr(g), _ptr(a), _ptr(A_log), _ptr(dt_bias)
    args.beta = _ptr(beta_t)
    args.h0, args.cu_seqlens = _ptr(h0), _ptr(cu_seqlens)
    args.o, args.hT, args.err = _ptr(o), _ptr(hT), _ptr(err)
    args.h_chunks = _ptr(h_chunks)
    return args


def chunk_workspace_size(args: ChunkArgs) -> int:
    return int(load().kda_chunk_workspace_size(ctypes.byref(args)))


def kda_chunk_fwd(q, k, v, *, scale, g=None, a=None, dt_bias=None, A_log=None, beta=None, b=None,
                  h0=None, cu_seqlens=None, l2norm_qk=False, delta=True, o=None, hT=None,
                  output_final_state=True, workspace=None, err=None, stream=None, g_head=None, h_chunks=None):
    """Chunkwise KDA forward through libkda (see include/kda.h for the contract).

    q, k [B, T, H, dk]; v [B, T, H, dv] (bf16 or fp32, same dtype). The gate is
    g (fp32 [B, T, H, dk]) or gate inputs a (fp32 [B, T, H*dk]) + dt_bias
    (fp32 [H*dk]) + A_log (fp32 [H]), or the Gated DeltaNet per-head gate g_head
    (fp32 [B, T, H]), or none (g = 0). beta [B, T, H] is given
    as values (beta=) or logits (b=). h0 / returned hT are fp32 [N, H, dv, dk].
    h_chunks (fp32 [chunk_count(...), H, dv, dk], bf16 only) receives the state
    entering every 16-token chunk when given.
    Returns (o, hT) with hT None when output_final_state is False.
    """
    lib = load()
    B, T, H, _ = q.shape
    if o is None:
        o = torch.empty(B, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if hT is None and output_final_state:
        hT = torch.empty(N, H, v.shape[-1], q.shape[-1], dtype=torch.float32, device=q.device)
    args = make_chunk_args(q, k, v, scale=scale, g=g, a=a, dt_bias=dt_bias, A_log=A_log, beta=beta, b=b,
                           h0=h0, cu_seqlens=cu_seqlens, l2norm_qk=l2norm_qk, delta=delta, o=o, hT=hT,
                           err=err, g_head=g_head, h_chunks=h_chunks)
    need = int(lib.kda_chunk_workspace_size(ctypes.byref(args)))
    with _on_device(q):
        if need == 0:
            st = lib.kda_chunk_fwd(ctypes.byref(args), None, 0, _stream_ptr(stream, q.device))
            raise KdaError(st if st != KDA_OK else KDA_ERR_INVALID_ARG, "kda_chunk_fwd")
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        st = lib.kda_chunk_fwd(ctypes.byref(args), ctypes.c_void_p(_ptr(workspace)), need,
                               _stream_ptr(stream, q.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd")
    return o, hT


def kda_chunk_fwd_noalloc(q, k, v, *, scale, g=None, a=None, dt_bias=None, A_log=None, beta=None, b=None,
                          h0=None, cu_seqlens=None, l2norm_qk=False, delta=True, o=None, hT=None,
                          output_final_state=True, err=None, stream=None, g_head=None, h_chunks=None):
    """kda_chunk_fwd on the library's own scratch buffer: the C call allocates
    nothing (for callers that may not allocate device memory; see
    include/kda.h). Outputs o / hT are allocated here with torch unless given.
    Raises KdaError(KDA_ERR_TOO_LARGE) when the request needs more than
    KDA_NOALLOC_SCRATCH_BYTES of scratch."""
    lib = load()
    B, T, H, _ = q.shape
    if o is None:
        o = torch.empty(B, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if hT is None and output_final_state:
        hT = torch.empty(N, H, v.shape[-1], q.shape[-1], dtype=torch.float32, device=q.device)
    args = make_chunk_args(q, k, v, scale=scale, g=g, a=a, dt_bias=dt_bias, A_log=A_log, beta=beta, b=b,
                           h0=h0, cu_seqlens=cu_seqlens, l2norm_qk=l2norm_qk, delta=delta, o=o, hT=hT,
                           err=err, g_head=g_head, h_chunks=h_chunks)
    with _on_device(q):
        st = lib.kda_chunk_fwd_noalloc(ctypes.byref(args), _stream_ptr(stream, q.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_noalloc")
    return o, hT


def make_decode_args(packed_qkv, a, b, A_log, dt_bias, state_pool, indices, *, H, HV, K, V, scale,
                     l2norm_qk=True, o=None, err=None, check_indices=False):
    args = DecodeArgs()
    args.B = packed_qkv.shape[0]
    args.H, args.HV, args.K, args.V = H, HV, K, V
    args.num_slots = state_pool.shape[0]
    args.flags = (KDA_FLAG_L2NORM_QK if l2norm_qk else 0) | (KDA_FLAG_CHECK_INDICES if check_indices else 0)
    args.scale = float(scale)
    args.packed_qkv, args.a, args.b = _ptr(packed_qkv), _ptr(a), _ptr(b)
    args.A_log, args.dt_bias = _ptr(A_log), _ptr(dt_bias)
    args.state_pool, args.indices = _ptr(state_pool), _ptr(indices)
    args.o, args.err = _ptr(o), _ptr(err)
    return args


def kda_decode_step(packed_qkv, a, b, A_log, dt_bias, state_pool, indices, *, H, HV, K, V, scale,
                    l2norm_qk=True, o=None, err=None, stream=None, check_indices=False):
    """Fused T=1 decode through libkda; state_pool is updated in place. Returns o [B, HV, V] bf16.
    check_indices (needs err): a debug check that the valid slot indices are distinct."""
    lib = load()
    if o is None:
        o = torch.empty(packed_qkv.shape[0], HV, V, dtype=torch.bfloat16, device=packed_qkv.device)
    args = make_decode_args(packed_qkv, a, b, A_log, dt_bias, state_pool, indices, H=H, HV=HV, K=K, V=V,
                            scale=scale, l2norm_qk=l2norm_qk, o=o, err=err, check_indices=check_indices)
    with _on_device(packed_qkv):
        st = lib.kda_decode_step(ctypes.byref(args), _stream_ptr(stream, packed_qkv.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_step")
    return o


def make_recurrent_args(q, k, v, a, b, A_log, dt_bias, state_pool, indices, *, scale, l2norm_qk=True,
                        o=None, err=None, check_indices=False):
    args = RecurrentArgs()
    args.B, args.T, args.H, args.K = (int(x) for x in q.shape)
    args.HV, args.V = int(v.shape[2]), int(v.shape[3])
    args.num_slots = state_pool.shape[0]
    args.flags = (KDA_FLAG_L2NORM_QK if l2norm_qk else 0) | (KDA_FLAG_CHECK_INDICES if check_indices else 0)
    args.scale = float(scale)
    args.q, args.k, args.v, args.a, args.b = _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b)
    args.A_log, args.dt_bias = _ptr(A_log), _ptr(dt_bias)
    args.state_pool, args.indices = _ptr(state_pool), _ptr(indices)
    args.o, args.err = _ptr(o), _ptr(err)
    return args


def kda_recurrent_step(q, k, v, a, b, A_log, dt_bias, state_pool, indices, *, scale, l2norm_qk=True,
                       o=None, err=None, stream=None, check_indices=False):
    """T tokens per row (q, k [B, T, H, K]; v [B, T, HV, V]; a [B, T, HV*K]; b [B, T, HV])
    through libkda on the slot pool, updated in place. Returns o [B, T, HV, V] bf16."""
    lib = load()
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], v.shape[3], dtype=torch.bfloat16, device=q.device)
    args = make_recurrent_args(q, k, v, a, b, A_log, dt_bias, state_pool, indices, scale=scale,
                               l2norm_qk=l2norm_qk, o=o, err=err, check_indices=check_indices)
    with _on_device(q):
        st = lib.kda_recurrent_step(ctypes.byref(args), _stream_ptr(stream, q.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_step")
    return o


def kda_head_rmsnorm(x, weight, *, eps, out=None, stream=None):
    """Per-head RMSNorm over the last axis (V) of x (bf16, any leading shape) with
    an fp32 weight [V]; out may be x itself. Returns out."""
    lib = load()
    if out is None:
        out = torch.empty_like(x)
    args = RmsNormArgs()
    args.V = int(x.shape[-1])
    args.R = int(x.numel() // max(args.V, 1))
    args.eps = float(eps)
    args.x, args.weight, args.y = _ptr(x), _ptr(weight), _ptr(out)
    with _on_device(x):
        st = lib.kda_head_rmsnorm(ctypes.byref(args), _stream_ptr(stream, x.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_head_rmsnorm")
    return out


def kda_decode_conv_step(mixed_qkv, conv_state_in, conv_weight, conv_bias, a, b, A_log, dt_bias, state_pool,
                         indices, *, H, HV, K, V, scale, conv_state_out=None, l2norm_qk=True, o=None, err=None,
                         stream=None, check_indices=False):
    """Decode with its causal conv1d + SiLU in front (see include/kda.h).
    mixed_qkv bf16 [B, C] is the conv input; conv_state_in bf16 [slots, W-1, C];
    conv_weight fp32 [C, W]; conv_bias fp32 [C] or None. conv_state_out defaults
    to conv_state_in (in place, allowed when HV == H). state_pool is updated in
    place. Returns o [B, HV, V] bf16."""
    lib = load()
    if o is None:
        o = torch.empty(mixed_qkv.shape[0], HV, V, dtype=torch.bfloat16, device=mixed_qkv.device)
    args = DecodeConvArgs()
    args.dec = make_decode_args(mixed_qkv, a, b, A_log, dt_bias, state_pool, indices, H=H, HV=HV, K=K, V=V,
                                scale=scale, l2norm_qk=l2norm_qk, o=o, err=err, check_indices=check_indices)
    args.W = int(conv_weight.shape[-1])
    args.conv_state_in = _ptr(conv_state_in)
    args.conv_state_out = _ptr(conv_state_in if conv_state_out is None else conv_state_out)
    args.conv_weight, args.conv_bias = _ptr(conv_weight), _ptr(conv_bias)
    with _on_device(mixed_qkv):
        st = lib.kda_decode_conv_step(ctypes.byref(args), _stream_ptr(stream, mixed_qkv.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_conv_step")
    return o


def chunk_count(B, T, cu_seqlens=None):
    """Number of 16-token chunks of a call: the first dimension of h_chunks."""
    if cu_seqlens is None:
        return B * ((T + 15) // 16)
    cu = cu_seqlens.detach().to("cpu").tolist()
    return sum((cu[i + 1] - cu[i] + 15) // 16 for i in range(len(cu) - 1))


def kda_chunk_output(q, k, v, h_chunks, *, scale, g=None, a=None, dt_bias=None, A_log=None, beta=None, b=None,
                     cu_seqlens=None, l2norm_qk=False, delta=True, o=None, workspace=None, err=None, stream=None,
                     g_head=None):
    """Chunk-parallel output pass: o from the inputs and the per-chunk entering
    states h_chunks that kda_chunk_fwd(h_chunks=...) wrote. Returns o."""
    lib = load()
    B, T, H, _ = q.shape
    if o is None:
        o = torch.empty(B, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
    args = make_chunk_args(q, k, v, scale=scale, g=g, a=a, dt_bias=dt_bias, A_log=A_log, beta=beta, b=b,
                           cu_seqlens=cu_seqlens, l2norm_qk=l2norm_qk, delta=delta, o=o, err=err, g_head=g_head,
                           h_chunks=h_chunks)
    need = int(lib.kda_chunk_workspace_size(ctypes.byref(args)))
    with _on_device(q):
        if need == 0:
            st = lib.kda_chunk_output(ctypes.byref(args), None, 0, _stream_ptr(stream, q.device))
            raise KdaError(st if st != KDA_OK else KDA_ERR_INVALID_ARG, "kda_chunk_output")
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        st = lib.kda_chunk_output(ctypes.byref(args), ctypes.c_void_p(_ptr(workspace)), need,
                                  _stream_ptr(stream, q.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_output")
    return o
