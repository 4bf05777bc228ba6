"""Plain fp64 CPU oracle for the KDA chunk forward, the fused T=1 decode step and
the short-T recurrent step on a state pool.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline legs of bench.py, never by the CUDA path (and it imports nothing
from it). Every function is pinned in tests/test_oracle_pins.py.

Sources (web pages, cited by title and section):

* [TL]   "TileLang 实战：KDA 从零到一--Chunked 线性注意力" (ggaaooppeenngg.github.io),
         §1 (the KDA recurrence and the five-level ladder), §2 (chunk identity),
         §3 (fp64 references), §6.4 (sequence kept out of the grid, d_v split).
* [LA]   "06 · linear 路线（一）：kernel trick、RNN 等价与三种计算形式"
         (llm-infra-atlas.github.io), §2 (RNN form), §3 (parallel / recurrent /
         chunkwise forms).
* [FKDA] "FlashKDA里的L矩阵和Mqk矩阵是什么" (lshu.cn), sections 背景 (token
         recurrence in delta form), L矩阵的构造, Mqk矩阵的构造, 为什么CHUNK=16
         (Neumann inverse), K2 内核如何消费 (chunk formulas).
* [PR]   sglang PR #26586 summary (prhub.com.cn), "关键源码片段": the packed
         decode kernel's behaviour (packed q|k|v row, L2 norm with eps 1e-6,
         gate -exp(A_log)*softplus(a+dt_bias), beta = sigmoid(b), pad slot -1,
         head grouping i_h = i_hv // (HV // H)).

Layouts (shared with the C ABI so that arrays can be compared directly):
  q, k      [T, H, K]   per sequence (the multi-sequence wrappers take [B, T, H, K])
  v, o      [T, H, V]
  g         [T, H, K]   log-decay per token and key channel (g <= 0)
  beta      [T, H]
  h0, hT    [H, V, K]   stored state, the transpose of the math state S[K, V]
The oracle works on the math state S[K, V] internally: S_t = S_{t-1} decayed on
its key rows, o_t = scale * S_t^T q_t ([TL] §1 gives the transposed (d_v, d_k)
form; [FKDA] 背景 gives the same recurrence with the state read as k^T S).

Readings of points the pages leave open:
  * softplus is the plain definition log(1 + e^x); kernels may switch to x above
    a threshold, the difference there is below 2.1e-9.
  * the L2 norm is x / sqrt(sum x^2 + 1e-6) ([PR] kernel source).
  * "delta term off" means u_t = v_t: beta is ignored and nothing is subtracted.
  * chunks restart at every sequence start; a last partial chunk is simply
    shorter (the GPU pads it, the oracle does not need to).
"""

from __future__ import annotations

import math

import numpy as np

L2NORM_EPS = 1e-6


# ----------------------------------------------------------------------------
# Elementwise pieces ([PR] decode kernel; [TL] §1 log-domain gate)
# ----------------------------------------------------------------------------

def l2_normalize(x: np.ndarray) -> np.ndarray:
    """x / sqrt(sum(x^2) + 1e-6) over the last axis ([PR], in-kernel q/k L2 norm)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2NORM_EPS)


def softplus(x: np.ndarray) -> np.ndarray:
    """log(1 + e^x), evaluated without overflow."""
    return np.logaddexp(0.0, np.asarray(x, dtype=np.float64))


def sigmoid(x: np.ndarray) -> np.ndarray:
    """1 / (1 + e^-x) ([PR]: beta = sigmoid(b))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def kda_gate(a: np.ndarray, dt_bias: np.ndarray, A_log: np.ndarray) -> np.ndarray:
    """Per-channel log-decay g = -exp(A_log[h]) * softplus(a + dt_bias[h, c]).

    [PR] "KDA per-K 门控": a is [..., H, K] (one value per head and key channel),
    dt_bias is [H, K], A_log is [H]. Returns g with the shape of a; g <= 0.
    """
    a = np.asarray(a, dtype=np.float64)
    dt_bias = np.asarray(dt_bias, dtype=np.float64)
    A_log = np.asarray(A_log, dtype=np.float64)
    return -np.exp(A_log)[:, None] * softplus(a + dt_bias)


def head_gate_to_channels(g_head: np.ndarray, K: int) -> np.ndarray:
    """Gated DeltaNet's gate: one log-decay per token and head, the same for every
    key channel ([TL] §1 ladder: Gated DeltaNet = scalar decay + delta rule, KDA
    refines it to per-channel; [LA] model tree: Mamba-2 / SSD scalar alpha_t).
    g_head [..., H] -> g [..., H, K]."""
    g_head = np.asarray(g_head, dtype=np.float64)
    return np.repeat(g_head[..., None], K, axis=-1)


# ----------------------------------------------------------------------------
# Token-by-token recurrence: the definition ([TL] §1, [FKDA] 背景)
# ----------------------------------------------------------------------------

def _token_step(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    """One token of KDA for all heads at once.

    S: [H, K, V] math state entering the token; q_t, k_t, g_t: [H, K];
    v_t: [H, V]; beta_t: [H]. Returns (S_t, o_t).

    S~  = diag(e^{g_t}) S                      (decay acts on the key index)
    u_t = beta_t (v_t - S~^T k_t)              (delta rule; u_t = v_t when off)
    S_t = S~ + k_t u_t^T
    o_t = scale * S_t^T q_t                    (read after the write)
    """
    S = np.exp(g_t)[:, :, None] * S
    if delta:
        read = np.einsum("hk,hkv->hv", k_t, S)
        u = beta_t[:, None] * (v_t - read)
    else:
        u = v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    o_t = scale * np.einsum("hk,hkv->hv", q_t, S)
    return S, o_t


def kda_recurrent(q, k, v, g, beta, scale, h0=None, delta=True):
    """Token recurrence for ONE sequence.

    q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H] (ignored when delta is off);
    h0: [H, V, K] stored state or None (zeros). Returns (o [T, H, V], hT [H, V, K]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    T, H, K = q.shape
    V = v.shape[-1]
    beta = np.zeros((T, H)) if beta is None else np.asarray(beta, np.float64)
    if h0 is None:
        S = np.zeros((H, K, V))
    else:
        S = np.array(np.asarray(h0, np.float64).transpose(0, 2, 1))
    o = np.zeros((T, H, V))
    for t in range(T):
        S, o[t] = _token_step(S, q[t], k[t], v[t], g[t], beta[t], scale, delta)
    return o, np.ascontiguousarray(S.transpose(0, 2, 1))


def _sequences(B, T, cu_seqlens):
    """(batch row, start, end) triples: B rows of length T, or the packed
    sequences of cu_seqlens over a single row."""
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    return [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def kda_forward(q, k, v, *, scale, g=None, a=None, dt_bias=None, A_log=None,
                beta=None, b=None, h0=None, cu_seqlens=None, l2norm_qk=False,
                delta=True, chunk_size=None, g_head=None, chunk_states=False):
    """The chunk-forward operation as the C ABI exposes it, computed in fp64.

    q, k: [B, T, H, K]; v: [B, T, H, V]. The gate is given either as g
    [B, T, H, K], or as gate inputs a [B, T, H*K], dt_bias [H*K], A_log [H]
    (g = -exp(A_log) * softplus(a + dt_bias)), or per head as g_head [B, T, H]
    (Gated DeltaNet: the same decay on every key channel), or not at all (g = 0).
    beta [B, T, H] is given directly or as logits b (beta = sigmoid(b)).
    h0: [N, H, V, K] or None. cu_seqlens: [N+1] over a single row (B == 1) or None.
    chunk_size None runs the token recurrence; an integer runs kda_chunked.
    Returns (o [B, T, H, V], hT [N, H, V, K]), and with chunk_states also the
    states entering every 16-token chunk, sequence after sequence
    ([sum_n ceil(len_n/16), H, V, K], chunk_start_states).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if l2norm_qk:
        q = l2_normalize(q)
        k = l2_normalize(k)
    if g is not None:
        g = np.asarray(g, np.float64)
    elif g_head is not None:
        g = head_gate_to_channels(g_head, K)
    elif a is not None:
        g = kda_gate(np.asarray(a, np.float64).reshape(B, T, H, K),
                     np.asarray(dt_bias, np.float64).reshape(H, K), A_log)
    else:
        g = np.zeros((B, T, H, K))
    if beta is None and b is not None:
        beta = sigmoid(b)
    beta = np.zeros((B, T, H)) if beta is None else np.asarray(beta, np.float64)
    seqs = _sequences(B, T, cu_seqlens)
    o = np.zeros((B, T, H, V))
    hT = np.zeros((len(seqs), H, V, K))
    snaps = []
    for n, (row, s, e) in enumerate(seqs):
        h0n = None if h0 is None else np.asarray(h0, np.float64)[n]
        args = (q[row, s:e], k[row, s:e], v[row, s:e], g[row, s:e], beta[row, s:e], scale)
        if chunk_size is None:
            o[row, s:e], hT[n] = kda_recurrent(*args, h0=h0n, delta=delta)
        else:
            o[row, s:e], hT[n] = kda_chunked(*args, C=chunk_size, h0=h0n, delta=delta)
        if chunk_states and e > s:
            snaps.append(chunk_start_states(*args, C=16, h0=h0n, delta=delta))
    if chunk_states:
        return o, hT, (np.concatenate(snaps) if snaps else np.zeros((0, H, V, K)))
    return o, hT


def chunk_start_states(q, k, v, g, beta, scale, C, h0=None, delta=True):
    """The state entering every C-token chunk of ONE sequence (stored layout
    [n_chunks, H, V, K]): snapshot 0 is h0, snapshot c the state after tokens
    0 .. cC-1. These are the per-chunk states a chunk-parallel output pass
    needs (the materialised h of [TL] §6 / [LA] §3.3's chunkwise form: inter-chunk
    recurrence first, then every chunk's output from its entering state)."""
    T = np.asarray(q).shape[0]
    H, K = np.asarray(q).shape[1:]
    V = np.asarray(v).shape[-1]
    n = (T + C - 1) // C
    out = np.zeros((n, H, V, K))
    state = np.zeros((H, V, K)) if h0 is None else np.asarray(h0, np.float64)
    for c in range(n):
        out[c] = state
        s, e = c * C, min(T, (c + 1) * C)
        _, state = kda_recurrent(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e] if beta is not None else None,
                                 scale, h0=state, delta=delta)
    return out


# ----------------------------------------------------------------------------
# Chunked form: L, Mqk, exact inverse ([FKDA]; [TL] §2; [LA] §3.3)
# ----------------------------------------------------------------------------

def chunk_matrices(q, k, g, beta, scale):
    """Intra-chunk quantities for one chunk of n tokens, all heads.

    q, k, g: [n, H, K]; beta: [n, H]. With G_i = sum_{j<=i} g_j (inclusive,
    per channel, restarting at the chunk start; [FKDA] L矩阵的构造):
      q_dec[i] = scale * q_i * e^{G_i}          k_dec[i] = k_i * e^{G_i}
      k_res[j] = k_j * e^{G_last - G_j}         gamma    = e^{G_last}
      L[i, j]  = beta_i * sum_c k_ic k_jc e^{G_ic - G_jc}       for j < i, else 0
      Mqk[i,j] = scale  * sum_c q_ic k_jc e^{G_ic - G_jc}       for j <= i, else 0
    The pair factors are exponentials of differences G_i - G_j <= 0, formed
    directly (never as a product of e^{G_i} and e^{-G_j}, which overflows).
    Returns a dict of arrays with a leading head axis: q_dec, k_dec, k_res
    [H, n, K], gamma [H, K], L, Mqk [H, n, n].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    n = q.shape[0]
    G = np.cumsum(g, axis=0)                             # [n, H, K]
    qh, kh, Gh = (x.transpose(1, 0, 2) for x in (q, k, G))  # [H, n, K]
    diff = Gh[:, :, None, :] - Gh[:, None, :, :]          # [H, i, j, K] = G_i - G_j
    lower_incl = np.tril(np.ones((n, n), dtype=bool))
    lower_strict = np.tril(np.ones((n, n), dtype=bool), -1)
    decay = np.exp(np.where(lower_incl[None, :, :, None], diff, -np.inf))
    kk = np.einsum("hic,hjc,hijc->hij", kh, kh, decay)
    qk = np.einsum("hic,hjc,hijc->hij", qh, kh, decay)
    L = np.where(lower_strict[None], beta.T[:, :, None] * kk, 0.0)
    Mqk = np.where(lower_incl[None], scale * qk, 0.0)
    G_last = Gh[:, -1, :]
    return {
        "q_dec": scale * qh * np.exp(Gh),
        "k_dec": kh * np.exp(Gh),
        "k_res": kh * np.exp(G_last[:, None, :] - Gh),
        "gamma": np.exp(G_last),
        "L": L,
        "Mqk": Mqk,
    }


def forward_substitution(L, R):
    """Solve (I + L) X = R for strictly lower-triangular L, row by row.

    Row i of X is R_i - sum_{j<i} L[i, j] X_j: the cascade of corrections that
    [FKDA] 背景 describes (each token's delta corrected by the earlier writes).
    L: [..., n, n]; R: [..., n, m].
    """
    L = np.asarray(L, np.float64)
    X = np.array(np.asarray(R, np.float64))
    n = L.shape[-1]
    for i in range(n):
        for j in range(i):
            X[..., i, :] -= L[..., i, j, None] * X[..., j, :]
    return X


def neumann_inverse(L):
    """(I + L)^{-1} by the Neumann series of X = -L, summed by repeated squaring.

    [FKDA] 为什么CHUNK=16: L is strictly lower, so L^n = 0 for n >= size and the
    finite series sum_{n<size} X^n is the exact inverse. For size 16 it is the
    product (I + X)(I + X^2)(I + X^4)(I + X^8): three squarings and three
    products. Sizes that are not a power of two use the next power of two.
    """
    L = np.asarray(L, np.float64)
    n = L.shape[-1]
    eye = np.broadcast_to(np.eye(n), L.shape)
    X = -L
    inv = eye + X
    P = X
    span = 2
    while span < n:
        P = P @ P
        inv = inv @ (eye + P)
        span *= 2
    return inv


def kda_chunked(q, k, v, g, beta, scale, C, h0=None, delta=True,
                solver="substitution"):
    """Chunked KDA for ONE sequence with chunk size C ([FKDA] 一句话总结, K2).

    For each chunk, with S the state entering it:
      U = (I + L)^{-1} (beta * (V - K_dec S))      (U = V when delta is off)
      O = Q_dec S + Mqk U
      S = diag(gamma) S + K_res^T U
    The sign convention: the pages print "(I - L)^{-1}" with the L of
    L矩阵的构造 carrying a stripped minus sign; derived from the token
    recurrence the correction is U_i = R_i - sum_{j<i} L_ij U_j, i.e. (I + L)^{-1}.
    solver: "substitution" (forward substitution) or "neumann".
    Returns (o [T, H, V], hT [H, V, K]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    T, H, K = q.shape
    V = v.shape[-1]
    beta = np.zeros((T, H)) if beta is None else np.asarray(beta, np.float64)
    S = np.zeros((H, K, V)) if h0 is None else np.array(np.asarray(h0, np.float64).transpose(0, 2, 1))
    o = np.zeros((T, H, V))
    for s in range(0, T, C):
        e = min(s + C, T)
        m = chunk_matrices(q[s:e], k[s:e], g[s:e], beta[s:e], scale)
        vh = v[s:e].transpose(1, 0, 2)                        # [H, n, V]
        if delta:
            R = beta[s:e].T[:, :, None] * (vh - m["k_dec"] @ S)
            if solver == "neumann":
                U = neumann_inverse(m["L"]) @ R
            else:
                U = forward_substitution(m["L"], R)
        else:
            U = vh
        o[s:e] = (m["q_dec"] @ S + m["Mqk"] @ U).transpose(1, 0, 2)
        S = m["gamma"][:, :, None] * S + m["k_res"].transpose(0, 2, 1) @ U
    return o, np.ascontiguousarray(S.transpose(0, 2, 1))


# ----------------------------------------------------------------------------
# Fused T=1 packed decode ([PR] 关键源码片段)
# ----------------------------------------------------------------------------

def kda_decode(packed_qkv, a, b, A_log, dt_bias, state_pool, indices, *,
               H, HV, K, V, scale, l2norm_qk=True):
    """One decode token per batch row, reading q|k|v from a packed row.

    packed_qkv: [B, 2*H*K + HV*V] laid out [q (H*K) | k (H*K) | v (HV*V)];
    a: [B, HV*K]; b: [B, HV]; A_log: [HV]; dt_bias: [HV*K];
    state_pool: [num_slots, HV, V, K] (stored layout); indices: [B] int, -1 = pad.
    Value head hv reads query/key head hv // (HV // H).
    Returns (o [B, HV, V], new_pool); the input pool is not modified. Pad rows
    get o = 0 and touch no state. Valid indices must be distinct.
    """
    packed = np.asarray(packed_qkv, np.float64)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    pool = np.array(np.asarray(state_pool, np.float64))
    idx = np.asarray(indices).astype(np.int64)
    Bn = packed.shape[0]
    valid = idx[idx >= 0]
    if len(set(valid.tolist())) != len(valid):
        raise ValueError("valid slot indices must be distinct")
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    group = HV // H
    o = np.zeros((Bn, HV, V))
    heads = np.arange(HV) // group
    q_all = packed[:, : H * K].reshape(Bn, H, K)[:, heads]
    k_all = packed[:, H * K: 2 * H * K].reshape(Bn, H, K)[:, heads]
    v_all = packed[:, 2 * H * K: 2 * H * K + HV * V].reshape(Bn, HV, V)
    g_all = kda_gate(a.reshape(Bn, HV, K), np.asarray(dt_bias, np.float64).reshape(HV, K), A_log)
    beta_all = sigmoid(b)
    for row in range(Bn):
        s = int(idx[row])
        if s < 0:
            continue
        q = q_all[row]
        k = k_all[row]
        if l2norm_qk:
            q = l2_normalize(q)
            k = l2_normalize(k)
        S = pool[s].transpose(0, 2, 1)                         # [HV, K, V]
        S, o[row] = _token_step(S, q, k, v_all[row], g_all[row], beta_all[row], scale, True)
        pool[s] = S.transpose(0, 2, 1)
    return o, pool


def kda_recurrent_pool(q, k, v, a, b, A_log, dt_bias, state_pool, indices, *,
                       scale, l2norm_qk=True):
    """T tokens per batch row on a state-slot pool: the general fused recurrent
    step that the packed decode specialises ([PR] 功能与动机 and 实现拆解: the
    packed kernel replaces the generic path for one token per row; speculative
    and extend steps run several). Same recurrence, gate, beta, L2 norm, head
    grouping and pad convention as kda_decode.

    q, k: [B, T, H, K]; v: [B, T, HV, V]; a: [B, T, HV*K]; b: [B, T, HV] (beta
    logits); A_log: [HV]; dt_bias: [HV*K]; state_pool: [num_slots, HV, V, K]
    (stored layout); indices: [B] int, -1 = pad. Value head hv reads query/key
    head hv // (HV // H). Tokens of a row are applied in order to its slot's
    state. Returns (o [B, T, HV, V], new_pool); the input pool is not modified.
    Pad rows get o = 0 and touch no state. Valid indices must be distinct.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    pool = np.array(np.asarray(state_pool, np.float64))
    idx = np.asarray(indices).astype(np.int64)
    Bn, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    valid = idx[idx >= 0]
    if len(set(valid.tolist())) != len(valid):
        raise ValueError("valid slot indices must be distinct")
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    heads = np.arange(HV) // (HV // H)
    g_all = kda_gate(a.reshape(Bn, T, HV, K), np.asarray(dt_bias, np.float64).reshape(HV, K), A_log)
    beta_all = sigmoid(b)
    o = np.zeros((Bn, T, HV, V))
    for row in range(Bn):
        s = int(idx[row])
        if s < 0:
            continue
        S = pool[s].transpose(0, 2, 1)                         # [HV, K, V]
        for t in range(T):
            qt = q[row, t][heads]
            kt = k[row, t][heads]
            if l2norm_qk:
                qt = l2_normalize(qt)
                kt = l2_normalize(kt)
            S, o[row, t] = _token_step(S, qt, kt, v[row, t], g_all[row, t], beta_all[row, t], scale, True)
        pool[s] = S.transpose(0, 2, 1)
    return o, pool


def head_rmsnorm(x, weight, eps):
    """Output-side per-head RMSNorm ([LA] §1 and §4 (3): GLA / GDN / KDA drop
    the linear-attention normaliser and put an RMSNorm on each head's output).
    The pages give no formula; the plain RMSNorm is taken: for every row (one
    token of one head) y = x / sqrt(mean(x^2) + eps) * weight, eps from the caller.
    x: [..., V]; weight: [V]. Returns y with the shape of x."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(weight, np.float64)


def silu(x):
    """x * sigmoid(x), the activation the decode path applies after the conv."""
    x = np.asarray(x, np.float64)
    return x * sigmoid(x)


def causal_conv1d_update(x, conv_state, weight, bias):
    """One step of a depthwise causal convolution per channel ([PR] "关键源码片段",
    KDAAttnBackend.forward_decode: causal_conv1d_update(mixed_qkv, conv_states,
    conv_weights, bias, activation="silu") runs before the packed decode).

    x: [C] new input; conv_state: [W-1, C] the previous W-1 inputs, oldest
    first; weight: [C, W] (tap W-1 multiplies the newest input); bias: [C] or
    None. Returns (y = silu(sum_i weight[:, i] * window[i] + bias), new_state)
    with window = [conv_state; x] and new_state = window[1:].
    """
    x = np.asarray(x, np.float64)
    window = np.concatenate([np.asarray(conv_state, np.float64), x[None]], axis=0)  # [W, C]
    pre = np.einsum("cw,wc->c", np.asarray(weight, np.float64), window)
    if bias is not None:
        pre = pre + np.asarray(bias, np.float64)
    return silu(pre), window[1:]


def kda_decode_conv(mixed_qkv, conv_state, conv_weight, conv_bias, a, b, A_log, dt_bias, state_pool,
                    indices, *, H, HV, K, V, scale, l2norm_qk=True):
    """The decode step with its conv in front: per valid row, causal_conv1d_update
    + SiLU of the packed [q | k | v] row on the row's slot of the conv-state pool,
    then kda_decode on the result. conv_state: [num_slots, W-1, C], C = 2*H*K +
    HV*V. Returns (o, new_state_pool, new_conv_state); inputs are not modified.
    Pad rows: o = 0, neither pool touched."""
    x = np.asarray(mixed_qkv, np.float64)
    cs = np.array(np.asarray(conv_state, np.float64))
    idx = np.asarray(indices).astype(np.int64)
    y = np.zeros_like(x)
    for row in range(x.shape[0]):
        s = int(idx[row])
        if s < 0:
            continue
        y[row], cs[s] = causal_conv1d_update(x[row], cs[s], conv_weight, conv_bias)
    o, pool = kda_decode(y, a, b, A_log, dt_bias, state_pool, indices, H=H, HV=HV, K=K, V=V, scale=scale,
                         l2norm_qk=l2norm_qk)
    return o, pool, cs


def default_scale(K: int) -> float:
    """K^-0.5, the scale the decode caller passes ([PR] head_k_dim ** -0.5)."""
    return 1.0 / math.sqrt(K)
