"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each pin is a plain function that raises AssertionError when the oracle breaks
it, so that test_mutants_are_caught can plant plausible mistakes in the oracle
(on the CPU) and check that some pin notices every one of them.

Sources: hand-worked fixtures under tests/golden/ (exact fractions), the
textbook linear-attention parallel form and chunk identity (TileLang 实战：KDA
从零到一 §2, §3; 06 · linear 路线（一） §3), the GLA / RetNet special cases of the
ladder (TileLang 实战 §1 table), the nilpotency of L and the Neumann inverse
(FlashKDA里的L矩阵和Mqk矩阵 §为什么CHUNK=16), the exact-write property of the delta
rule with unit keys (06 · linear 路线（一） §4 (2): the regression objective), and
brute force on tiny inputs.
"""

import json
import math
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

from oracle import kda_oracle as ko

GOLDEN = Path(__file__).parent / "golden"


def _frac(x):
    return np.vectorize(lambda s: float(Fraction(s)), otypes=[np.float64])(np.array(x, dtype=object))


def _rng(seed):
    return np.random.default_rng(seed)


def _rel(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300))


def _rand_case(seed, T=13, H=2, K=4, V=5, gate=True, beta=True, h0=True):
    r = _rng(seed)
    q = r.standard_normal((T, H, K))
    k = ko.l2_normalize(r.standard_normal((T, H, K)))
    v = r.standard_normal((T, H, V))
    g = -r.uniform(0.0, 1.5, (T, H, K)) if gate else np.zeros((T, H, K))
    b = r.uniform(0.0, 1.0, (T, H)) if beta else np.ones((T, H))
    s0 = 0.3 * r.standard_normal((H, V, K)) if h0 else None
    return q, k, v, g, b, s0


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------

def pin_hand_worked_chunk():
    """Exact fractions worked by hand (tests/golden/hand_worked_chunk.json)."""
    d = json.loads((GOLDEN / "hand_worked_chunk.json").read_text())
    q, k, v = _frac(d["q"]), _frac(d["k"]), _frac(d["v"])
    g = np.log(_frac(d["alpha"]))
    beta = _frac(d["beta"])
    h0 = _frac(d["h0"])
    scale = float(Fraction(d["scale"]))
    for key, delta in (("delta_on", True), ("delta_off", False)):
        o_exp = _frac(d[key]["o"])
        h_exp = _frac(d[key]["hT"])
        o, hT = ko.kda_recurrent(q, k, v, g, beta, scale, h0=h0, delta=delta)
        np.testing.assert_allclose(o, o_exp, rtol=0, atol=1e-13)
        np.testing.assert_allclose(hT, h_exp, rtol=0, atol=1e-13)
        for C in (1, 2, 3):
            oc, hc = ko.kda_chunked(q, k, v, g, beta, scale, C, h0=h0, delta=delta)
            np.testing.assert_allclose(oc, o_exp, rtol=0, atol=1e-13)
            np.testing.assert_allclose(hc, h_exp, rtol=0, atol=1e-13)


def pin_level1_quadratic_form():
    """g = 0, delta off: o = scale (tril(Q K^T) V + Q S0), the parallel form of
    causal linear attention (06 · linear 路线（一） §3.1), with a nonzero S0."""
    r = _rng(1)
    B, T, H, K, V = 2, 12, 2, 4, 4           # the worked example sizes of TileLang 实战 §3.4
    q, k, v = (r.standard_normal((B, T, H, d)) for d in (K, K, V))
    h0 = r.standard_normal((B, H, V, K))
    scale = 0.7
    o, hT = ko.kda_forward(q, k, v, scale=scale, h0=h0, delta=False)
    for b in range(B):
        for h in range(H):
            Q, Kk, Vv = q[b, :, h], k[b, :, h], v[b, :, h]
            S0 = h0[b, h].T
            ref = scale * (np.tril(Q @ Kk.T) @ Vv + Q @ S0)
            assert _rel(o[b, :, h], ref) < 1e-13
            assert _rel(hT[b, h], (S0 + Kk.T @ Vv).T) < 1e-13


def pin_level1_chunk_identity():
    """O_c = Q_c S_prev + tril(Q_c K_c^T) V_c with S_prev from a right-shifted
    cumsum of per-chunk K^T V (TileLang 实战 §2.1 and reference B of §3.2)."""
    r = _rng(2)
    B, T, H, D, BC = 2, 12, 2, 4, 4
    q, k, v = (r.standard_normal((B, T, H, D)) for _ in range(3))
    o, _ = ko.kda_forward(q, k, v, scale=1.0, delta=False)
    NC = T // BC
    for b in range(B):
        for h in range(H):
            Qc = q[b, :, h].reshape(NC, BC, D)
            Kc = k[b, :, h].reshape(NC, BC, D)
            Vc = v[b, :, h].reshape(NC, BC, D)
            states = np.cumsum(np.einsum("cnd,cnv->cdv", Kc, Vc), axis=0)
            prev = np.concatenate([np.zeros((1, D, D)), states[:-1]], axis=0)
            ref = np.einsum("cnd,cdv->cnv", Qc, prev) + np.tril(np.einsum("cnd,cmd->cnm", Qc, Kc)) @ Vc
            assert _rel(o[b, :, h], ref.reshape(T, D)) < 1e-13


def pin_gla_parallel_form():
    """Gated, delta off (ladder level 3): explicit double sum
    o_i = scale sum_{j<=i} (sum_c q_ic k_jc e^{G_ic - G_jc}) v_j + scale (q_i e^{G_i})^T S0."""
    q, k, v, g, _, h0 = _rand_case(3, T=9, H=2, K=3, V=4)
    scale = 0.5
    o, _ = ko.kda_recurrent(q, k, v, g, None, scale, h0=h0, delta=False)
    G = np.cumsum(g, axis=0)
    T, H, K = q.shape
    ref = np.zeros_like(o)
    for h in range(H):
        S0 = h0[h].T
        for i in range(T):
            acc = (q[i, h] * np.exp(G[i, h])) @ S0
            for j in range(i + 1):
                w = sum(q[i, h, c] * k[j, h, c] * math.exp(G[i, h, c] - G[j, h, c]) for c in range(K))
                acc = acc + w * v[j, h]
            ref[i, h] = scale * acc
    assert _rel(o, ref) < 1e-13


def pin_retnet_scalar_decay():
    """Ladder level 2: one scalar gamma for every channel and token gives
    o = ((Q K^T) * Gamma) V with Gamma_ij = gamma^(i-j) for j <= i."""
    r = _rng(4)
    T, H, K, V = 10, 1, 3, 2
    q, k, v = r.standard_normal((T, H, K)), r.standard_normal((T, H, K)), r.standard_normal((T, H, V))
    gamma = 0.8
    g = np.full((T, H, K), math.log(gamma))
    o, _ = ko.kda_recurrent(q, k, v, g, None, 1.0, delta=False)
    i, j = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
    Gam = np.where(j <= i, gamma ** np.maximum(i - j, 0), 0.0)
    ref = ((q[:, 0] @ k[:, 0].T) * Gam) @ v[:, 0]
    assert _rel(o[:, 0], ref) < 1e-13


def pin_chunked_equals_recurrent():
    """The chunk form at C = 1, 4, 16 equals the token form (06 · linear 路线（一）
    §3.3: C interpolates between the recurrent and parallel forms), on ragged
    lengths and packed sequences."""
    q, k, v, g, b, h0 = _rand_case(5, T=37, H=2, K=6, V=5)
    scale = 0.4
    o_ref, h_ref = ko.kda_recurrent(q, k, v, g, b, scale, h0=h0)
    for C in (1, 4, 16):
        for solver in ("substitution", "neumann"):
            o, h = ko.kda_chunked(q, k, v, g, b, scale, C, h0=h0, solver=solver)
            assert _rel(o, o_ref) < 1e-12 and _rel(h, h_ref) < 1e-12
    # packed varlen through the ABI-shaped wrapper
    r = _rng(6)
    cu = np.array([0, 5, 21, 22, 40])
    Tt, H, K, V = 40, 2, 4, 3
    Q, Kk, Vv = r.standard_normal((1, Tt, H, K)), r.standard_normal((1, Tt, H, K)), r.standard_normal((1, Tt, H, V))
    a = r.standard_normal((1, Tt, H * K))
    dt = r.uniform(-1, 1, H * K)
    al = r.uniform(0, 1, H)
    bl = r.standard_normal((1, Tt, H))
    H0 = r.standard_normal((4, H, V, K))
    kw = dict(scale=0.3, a=a, dt_bias=dt, A_log=al, b=bl, h0=H0, cu_seqlens=cu, l2norm_qk=True)
    o1, h1 = ko.kda_forward(Q, Kk, Vv, **kw)
    o2, h2 = ko.kda_forward(Q, Kk, Vv, chunk_size=16, **kw)
    assert _rel(o2, o1) < 1e-12 and _rel(h2, h1) < 1e-12


def pin_L_nilpotent_and_inverse():
    """L^16 = 0 exactly; the Neumann product equals forward substitution and
    the library solve; (I + L) INV = I (FlashKDA §为什么CHUNK=16)."""
    r = _rng(7)
    n, H, K = 16, 3, 8
    q = r.standard_normal((n, H, K))
    k = ko.l2_normalize(r.standard_normal((n, H, K)))
    g = -r.uniform(0, 0.3, (n, H, K))
    beta = r.uniform(0.2, 1.0, (n, H))
    m = ko.chunk_matrices(q, k, g, beta, 0.5)
    L = m["L"]
    assert np.all(np.triu(L) == 0.0)
    P = np.broadcast_to(np.eye(n), L.shape).copy()
    for _ in range(16):
        P = P @ L
    assert np.all(P == 0.0)
    inv = ko.neumann_inverse(L)
    eye = np.broadcast_to(np.eye(n), L.shape)
    fs = ko.forward_substitution(L, eye)
    assert np.max(np.abs(inv - fs)) < 1e-13
    assert np.max(np.abs((eye + L) @ inv - eye)) < 1e-13
    R = r.standard_normal((H, n, 5))
    np.testing.assert_allclose(ko.forward_substitution(L, R), np.linalg.solve(eye + L, R), rtol=0, atol=1e-12)
    # sizes that are not a power of two
    for nn in (3, 5, 12):
        Ls = np.tril(r.standard_normal((nn, nn)), -1) * 0.5
        np.testing.assert_allclose(ko.neumann_inverse(Ls), np.linalg.inv(np.eye(nn) + Ls), rtol=0, atol=1e-10)


def pin_chunk_matrices_brute_force():
    """Every entry of L, Mqk and the decayed operands, brute force from the
    definitions in FlashKDA §L矩阵的构造 / §Mqk矩阵的构造."""
    r = _rng(8)
    n, H, K = 5, 1, 3
    q, k = r.standard_normal((n, H, K)), r.standard_normal((n, H, K))
    g = -r.uniform(0, 2, (n, H, K))
    beta = r.uniform(0, 1, (n, H))
    scale = 0.3
    m = ko.chunk_matrices(q, k, g, beta, scale)
    G = np.cumsum(g[:, 0], axis=0)
    for i in range(n):
        for j in range(n):
            s_kk = sum(k[i, 0, c] * k[j, 0, c] * math.exp(G[i, c] - G[j, c]) for c in range(K))
            s_qk = sum(q[i, 0, c] * k[j, 0, c] * math.exp(G[i, c] - G[j, c]) for c in range(K))
            assert math.isclose(m["L"][0, i, j], beta[i, 0] * s_kk if j < i else 0.0, abs_tol=1e-14)
            assert math.isclose(m["Mqk"][0, i, j], scale * s_qk if j <= i else 0.0, abs_tol=1e-14)
        for c in range(K):
            assert math.isclose(m["q_dec"][0, i, c], scale * q[i, 0, c] * math.exp(G[i, c]), rel_tol=1e-14)
            assert math.isclose(m["k_dec"][0, i, c], k[i, 0, c] * math.exp(G[i, c]), rel_tol=1e-14)
            assert math.isclose(m["k_res"][0, i, c], k[i, 0, c] * math.exp(G[-1, c] - G[i, c]), rel_tol=1e-14)
    np.testing.assert_allclose(m["gamma"][0], np.exp(G[-1]), rtol=1e-14)
    # large gates: exponentials of differences stay finite where e^{-G_j} overflows
    g_big = np.full((16, 1, 2), -40.0)
    mb = ko.chunk_matrices(np.ones((16, 1, 2)), np.ones((16, 1, 2)), g_big, np.ones((16, 1)), 1.0)
    assert np.all(np.isfinite(mb["L"])) and math.isclose(mb["L"][0, 15, 14], 2 * math.exp(-40.0), rel_tol=1e-12)


def pin_delta_exact_write():
    """beta = 1, g = 0, |k| = 1: after the write S_t^T k_t = v_t exactly (the
    delta rule minimises 1/2 |S^T k - v|^2; 06 · linear 路线（一） §4 (2)). Reading
    with q = k and scale = 1 therefore returns v_t at every step."""
    r = _rng(9)
    T, H, K, V = 20, 2, 8, 5
    k = r.standard_normal((T, H, K))
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, V))
    h0 = r.standard_normal((H, V, K))
    o, _ = ko.kda_recurrent(k, k, v, np.zeros((T, H, K)), np.ones((T, H)), 1.0, h0=h0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def pin_beta_zero_pure_decay():
    """beta = 0 (delta on): nothing is written, the state only decays:
    hT = h0 e^{sum g} on the key axis, o_t = scale (diag(e^{G_t}) S0)^T q_t."""
    q, k, v, g, _, h0 = _rand_case(10, T=11, H=2, K=4, V=3)
    scale = 0.9
    o, hT = ko.kda_recurrent(q, k, v, g, np.zeros(q.shape[:2]), scale, h0=h0)
    G = np.cumsum(g, axis=0)
    np.testing.assert_allclose(hT, h0 * np.exp(G[-1])[:, None, :], rtol=1e-13, atol=0)
    ref = scale * np.einsum("thk,hvk->thv", q * np.exp(G), h0)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-14)


def pin_orthonormal_keys():
    """k_t = e_{pi(t)}, beta = 1, g = 0: each token overwrites key row pi(t)
    of the math state with v_t; everything else is untouched."""
    r = _rng(11)
    T, H, K, V = 6, 1, 8, 3
    perm = r.permutation(K)[:T]
    k = np.zeros((T, H, K))
    for t in range(T):
        k[t, 0, perm[t]] = 1.0
    q = r.standard_normal((T, H, K))
    v = r.standard_normal((T, H, V))
    h0 = r.standard_normal((H, V, K))
    o, hT = ko.kda_recurrent(q, k, v, np.zeros((T, H, K)), np.ones((T, H)), 1.0, h0=h0)
    S = h0[0].T.copy()
    for t in range(T):
        S[perm[t]] = v[t, 0]
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(hT[0], S.T, rtol=0, atol=1e-13)


def pin_gate_sigmoid_l2norm():
    """Closed forms of the gate, sigmoid and L2 norm (tests/golden/gate_closed_forms.json)."""
    d = json.loads((GOLDEN / "gate_closed_forms.json").read_text())
    for c in d["gate_cases"]:
        g = ko.kda_gate(np.array([[c["x"]]]), np.zeros((1, 1)), np.array([c["A_log"]]))
        assert math.isclose(float(g[0, 0]), c["g"], rel_tol=1e-14, abs_tol=1e-15)
    for c in d["sigmoid_cases"]:
        assert math.isclose(float(ko.sigmoid(np.array(c["b"]))), c["beta"], rel_tol=1e-14)
    g = ko.kda_gate(np.array([[0.3, -0.2]]), np.array([[0.1, 0.5]]), np.array([0.7]))
    np.testing.assert_allclose(g, -math.exp(0.7) * np.log1p(np.exp(np.array([[0.4, 0.3]]))), rtol=1e-14)
    x = _rng(12).standard_normal((7, 9))
    y = ko.l2_normalize(x)
    s = np.sum(x * x, axis=-1)
    np.testing.assert_allclose(np.sum(y * y, axis=-1), s / (s + 1e-6), rtol=1e-14)
    np.testing.assert_allclose(y / x, (1 / np.sqrt(s + 1e-6))[:, None] * np.ones_like(x), rtol=1e-14)


def pin_decode_golden():
    """Hand-worked packed decode (tests/golden/hand_worked_decode.json): values,
    pad row, untouched slots."""
    d = json.loads((GOLDEN / "hand_worked_decode.json").read_text())
    pool_in = _frac(d["state_pool"])
    o, pool = ko.kda_decode(
        _frac(d["packed_qkv"]), _frac(d["a"]), _frac(d["b"]), _frac(d["A_log"]), _frac(d["dt_bias"]),
        pool_in, np.array(d["indices"]), H=d["H"], HV=d["HV"], K=d["K"], V=d["V"],
        scale=float(Fraction(d["scale"])))
    tol = d["tolerance"]
    np.testing.assert_allclose(o, _frac(d["expected_o"]), rtol=0, atol=tol)
    np.testing.assert_allclose(pool, _frac(d["expected_pool"]), rtol=0, atol=tol)
    assert np.all(o[1] == 0.0)
    assert np.array_equal(pool[0], pool_in[0])


def pin_decode_head_grouping():
    """HV = 2 H: value heads 2h and 2h+1 both read q/k head h. Running the same
    problem as two HV = H problems with repacked rows must give the same result."""
    r = _rng(13)
    B, H, HV, K, V = 3, 2, 4, 4, 3
    packed = r.standard_normal((B, 2 * H * K + HV * V))
    a = r.standard_normal((B, HV * K))
    bb = r.standard_normal((B, HV))
    A_log = r.uniform(0, 1, HV)
    dt = r.uniform(-1, 1, HV * K)
    pool = r.standard_normal((5, HV, V, K))
    idx = np.array([4, -1, 1])
    o, newp = ko.kda_decode(packed, a, bb, A_log, dt, pool, idx, H=H, HV=HV, K=K, V=V, scale=0.5)
    qs = packed[:, :H * K].reshape(B, H, K)
    ks = packed[:, H * K:2 * H * K].reshape(B, H, K)
    vs = packed[:, 2 * H * K:].reshape(B, HV, V)
    for hv in range(HV):
        h = hv // (HV // H)
        p1 = np.concatenate([qs[:, h], ks[:, h], vs[:, hv]], axis=1)
        o1, n1 = ko.kda_decode(p1, a[:, hv * K:(hv + 1) * K], bb[:, hv:hv + 1], A_log[hv:hv + 1],
                               dt[hv * K:(hv + 1) * K], pool[:, hv:hv + 1], idx, H=1, HV=1, K=K, V=V, scale=0.5)
        np.testing.assert_allclose(o[:, hv], o1[:, 0], rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(newp[:, hv], n1[:, 0], rtol=1e-14, atol=1e-14)


def pin_split_sequence():
    """Running T tokens equals running T1 tokens, then T - T1 from the state
    returned (the recurrent state is the whole carried context)."""
    q, k, v, g, b, h0 = _rand_case(14, T=29, H=2, K=4, V=4)
    o, h = ko.kda_recurrent(q, k, v, g, b, 0.6, h0=h0)
    for T1 in (1, 16, 17):
        o1, h1 = ko.kda_recurrent(q[:T1], k[:T1], v[:T1], g[:T1], b[:T1], 0.6, h0=h0)
        o2, h2 = ko.kda_chunked(q[T1:], k[T1:], v[T1:], g[T1:], b[T1:], 0.6, 16, h0=h1)
        assert _rel(np.concatenate([o1, o2]), o) < 1e-12 and _rel(h2, h) < 1e-12


def pin_value_split_invariance():
    """Value columns are independent (TileLang 实战 §6.4.1: d_v is a free
    dimension of every contraction): a column subset gives the same columns."""
    q, k, v, g, b, h0 = _rand_case(15, T=17, H=2, K=4, V=6)
    o, h = ko.kda_recurrent(q, k, v, g, b, 0.6, h0=h0)
    for cols in (slice(0, 2), slice(2, 6), slice(3, 4)):
        o2, h2 = ko.kda_recurrent(q, k, v[..., cols], g, b, 0.6, h0=h0[:, cols])
        np.testing.assert_allclose(o2, o[..., cols], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(h2, h[:, cols], rtol=1e-14, atol=1e-15)


def pin_recurrent_pool_is_repeated_decode():
    """T tokens per row on the pool equal T successive packed decode steps, each
    fed the pool the previous one returned (the recurrent step is the decode
    step applied token by token), with HV = 2 H grouping and a pad row."""
    r = _rng(16)
    B, T, H, HV, K, V = 3, 4, 2, 4, 4, 3
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K))
    v = r.standard_normal((B, T, HV, V))
    a = r.standard_normal((B, T, HV * K))
    bb = r.standard_normal((B, T, HV))
    A_log = r.uniform(0, 1, HV)
    dt = r.uniform(-1, 1, HV * K)
    pool = r.standard_normal((5, HV, V, K))
    idx = np.array([3, -1, 0])
    o, newp = ko.kda_recurrent_pool(q, k, v, a, bb, A_log, dt, pool, idx, scale=0.5)
    p = pool
    for t in range(T):
        packed = np.concatenate([q[:, t].reshape(B, -1), k[:, t].reshape(B, -1), v[:, t].reshape(B, -1)], axis=1)
        ot, p = ko.kda_decode(packed, a[:, t], bb[:, t], A_log, dt, p, idx, H=H, HV=HV, K=K, V=V, scale=0.5)
        np.testing.assert_allclose(o[:, t], ot, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(newp, p, rtol=1e-13, atol=1e-14)
    assert np.all(o[1] == 0.0) and np.array_equal(newp[1], pool[1])


def pin_recurrent_pool_tokens_matter():
    """Swapping two tokens of a row changes the result (the steps do not
    commute), and a one-token call equals the decode golden's row layout."""
    r = _rng(17)
    B, T, H, K, V = 1, 3, 1, 4, 4
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K))
    v = r.standard_normal((B, T, H, V))
    a = r.standard_normal((B, T, H * K))
    bb = r.standard_normal((B, T, H))
    pool = r.standard_normal((2, H, V, K))
    args = (r.uniform(0, 1, H), r.uniform(-1, 1, H * K), pool, np.array([1]))
    o, p = ko.kda_recurrent_pool(q, k, v, a, bb, *args, scale=0.5)
    perm = [1, 0, 2]
    o2, p2 = ko.kda_recurrent_pool(q[:, perm], k[:, perm], v[:, perm], a[:, perm], bb[:, perm], *args, scale=0.5)
    assert _rel(p2, p) > 1e-3 and _rel(o2[:, 2], o[:, 2]) > 1e-3


def pin_head_gate_semiseparable():
    """Gated DeltaNet's scalar decay with the delta term off is the
    semiseparable (Mamba-2 / SSD) form: o_t = scale [ (prod_{r<=t} a_r) S0^T q_t
    + sum_{s<=t} (prod_{s<r<=t} a_r) (q_t . k_s) v_s ], a_r = e^{g_r}; brute force
    over all (s, t) pairs. With the delta term on it must equal KDA whose
    per-channel gate repeats the head's value on every channel."""
    r = _rng(18)
    T, H, K, V = 9, 2, 3, 2
    q = r.standard_normal((1, T, H, K))
    k = r.standard_normal((1, T, H, K))
    v = r.standard_normal((1, T, H, V))
    gh = -r.uniform(0.05, 1.0, (1, T, H))
    h0 = r.standard_normal((1, H, V, K))
    o, hT = ko.kda_forward(q, k, v, scale=0.7, g_head=gh, h0=h0, delta=False)
    for h in range(H):
        S = h0[0, h].T.copy()                       # math state [K, V]
        for t in range(T):
            want = math.exp(gh[0, :t + 1, h].sum()) * (h0[0, h] @ q[0, t, h])
            for s in range(t + 1):
                want = want + math.exp(gh[0, s + 1:t + 1, h].sum()) * (q[0, t, h] @ k[0, s, h]) * v[0, s, h]
            np.testing.assert_allclose(o[0, t, h], 0.7 * want, rtol=1e-12, atol=1e-12)
        S = math.exp(gh[0, :, h].sum()) * S + sum(math.exp(gh[0, s + 1:, h].sum()) * np.outer(k[0, s, h], v[0, s, h])
                                                for s in range(T))
        np.testing.assert_allclose(hT[0, h], S.T, rtol=1e-12, atol=1e-12)
    bb = r.uniform(0, 1, (1, T, H))
    o1, h1 = ko.kda_forward(q, k, v, scale=0.7, g_head=gh, h0=h0, beta=bb)
    o2, h2 = ko.kda_forward(q, k, v, scale=0.7, g=np.repeat(gh[..., None], K, axis=-1), h0=h0, beta=bb)
    np.testing.assert_allclose(o1, o2, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(h1, h2, rtol=1e-14, atol=1e-14)


def pin_head_rmsnorm():
    """Hand-worked rows: [3, 4] has mean square 25/2, so with eps = 0 and weight
    [1, 2] the result is [3, 8] * sqrt(2) / 5; [1, 1] with eps = 1/2 gives
    weight / sqrt(3/2); a zero row stays zero. With unit weight and eps = 0 every
    nonzero row comes out with unit mean square, whatever its scale."""
    y = ko.head_rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(y, [[3 * math.sqrt(2) / 5, 8 * math.sqrt(2) / 5]], rtol=1e-15)
    y = ko.head_rmsnorm(np.array([[1.0, 1.0], [0.0, 0.0]]), np.array([0.5, -3.0]), 0.5)
    np.testing.assert_allclose(y[0], np.array([0.5, -3.0]) / math.sqrt(1.5), rtol=1e-15)
    assert np.all(y[1] == 0.0)
    x = _rng(19).standard_normal((5, 7)) * np.array([[1e-3], [1.0], [30.0], [2.0], [1e3]])
    y = ko.head_rmsnorm(x, np.ones(7), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(y, ko.head_rmsnorm(4.5 * x, np.ones(7), 0.0), rtol=1e-13)


def pin_conv1d_update_is_causal_convolution():
    """Stepping causal_conv1d_update through a sequence equals numpy's full
    convolution of each channel with its (reversed-tap) kernel, truncated to the
    causal part, then SiLU; an impulse history returns the taps; SiLU(x) =
    x / (1 + e^{-x})."""
    r = _rng(20)
    C, W, T = 5, 4, 11
    x = r.standard_normal((T, C))
    w = r.standard_normal((C, W))
    bias = r.standard_normal(C)
    state = np.zeros((W - 1, C))
    ys = []
    for t in range(T):
        y, state = ko.causal_conv1d_update(x[t], state, w, bias)
        ys.append(y)
    for c in range(C):
        full = np.convolve(x[:, c], w[c, ::-1])[:T] + bias[c]
        np.testing.assert_allclose(np.array(ys)[:, c], full / (1 + np.exp(-full)), rtol=1e-13, atol=1e-14)
    imp = np.zeros((W - 1, C))
    imp[0] = 1.0
    y, _ = ko.causal_conv1d_update(np.zeros(C), imp, w, None)
    pre = w[:, 0]
    np.testing.assert_allclose(y, pre / (1 + np.exp(-pre)), rtol=1e-14)


def pin_decode_conv_state_and_pads():
    """After W-1 decode steps with the conv in front, a valid row's conv state
    holds exactly its last W-1 inputs (whatever it started as); pad rows get
    o = 0 and leave both pools alone; a valid row's output matches decoding the
    SiLU of the causal convolution over its full input history."""
    r = _rng(21)
    B, H, HV, K, V, W, slots = 3, 1, 2, 4, 3, 3, 4
    C = 2 * H * K + HV * V
    w = r.standard_normal((C, W))
    bias = r.standard_normal(C)
    cs0 = r.standard_normal((slots, W - 1, C))
    pool = r.standard_normal((slots, HV, V, K))
    idx = np.array([2, -1, 0])
    A_log, dt = r.uniform(0, 1, HV), r.uniform(-1, 1, HV * K)
    xs = [r.standard_normal((B, C)) for _ in range(W - 1)]
    cs, p = cs0, pool
    for x in xs:
        a, bb = r.standard_normal((B, HV * K)), r.standard_normal((B, HV))
        o, p, cs = ko.kda_decode_conv(x, cs, w, bias, a, bb, A_log, dt, p, idx, H=H, HV=HV, K=K, V=V, scale=0.5)
        assert np.all(o[1] == 0.0)
    for row, s in ((0, 2), (2, 0)):
        np.testing.assert_array_equal(cs[s], np.stack([x[row] for x in xs]))
    for s in (1, 3):
        np.testing.assert_array_equal(cs[s], cs0[s])
        np.testing.assert_array_equal(p[s], pool[s])
    # one more step from a zero history: the output is the decode of SiLU(w[:, -1] x + bias)
    x = r.standard_normal((B, C))
    a, bb = r.standard_normal((B, HV * K)), r.standard_normal((B, HV))
    o, _, _ = ko.kda_decode_conv(x, np.zeros_like(cs0), w, bias, a, bb, A_log, dt, pool, idx, H=H, HV=HV, K=K, V=V,
                                 scale=0.5)
    pre = w[:, -1] * x + bias
    o2, _ = ko.kda_decode(pre / (1 + np.exp(-pre)), a, bb, A_log, dt, pool, idx, H=H, HV=HV, K=K, V=V, scale=0.5)
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-14)


def pin_chunk_start_states():
    """Snapshot 0 is h0; running each chunk alone from its snapshot reproduces
    that chunk's outputs of the whole-sequence run and lands on the next
    snapshot (the last one leads to hT): outputs are chunk-parallel given the
    snapshots."""
    q, k, v, g, b, h0 = _rand_case(22, T=37, H=2, K=4, V=3)
    o, hT = ko.kda_recurrent(q, k, v, g, b, 0.6, h0=h0)
    snaps = ko.chunk_start_states(q, k, v, g, b, 0.6, 16, h0=h0)
    assert snaps.shape == (3, 2, 3, 4)
    np.testing.assert_array_equal(snaps[0], h0)
    for c in range(3):
        s, e = 16 * c, min(37, 16 * (c + 1))
        oc, hc = ko.kda_recurrent(q[s:e], k[s:e], v[s:e], g[s:e], b[s:e], 0.6, h0=snaps[c])
        assert _rel(oc, o[s:e]) < 1e-12
        assert _rel(hc, snaps[c + 1] if c < 2 else hT) < 1e-12


PINS = [
    pin_hand_worked_chunk, pin_level1_quadratic_form, pin_level1_chunk_identity,
    pin_gla_parallel_form, pin_retnet_scalar_decay, pin_chunked_equals_recurrent,
    pin_L_nilpotent_and_inverse, pin_chunk_matrices_brute_force, pin_delta_exact_write,
    pin_beta_zero_pure_decay, pin_orthonormal_keys, pin_gate_sigmoid_l2norm,
    pin_decode_golden, pin_decode_head_grouping, pin_split_sequence, pin_value_split_invariance,
    pin_recurrent_pool_is_repeated_decode, pin_recurrent_pool_tokens_matter, pin_head_gate_semiseparable,
    pin_head_rmsnorm, pin_conv1d_update_is_causal_convolution, pin_decode_conv_state_and_pads,
    pin_chunk_start_states,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# Planted mistakes: each must break at least one pin
# ---------------------------------------------------------------------------

def _step_decay_after_write(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    read = np.einsum("hk,hkv->hv", k_t, S)
    u = beta_t[:, None] * (v_t - read) if delta else v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    S = np.exp(g_t)[:, :, None] * S
    return S, scale * np.einsum("hk,hkv->hv", q_t, S)


def _step_read_before_write(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    S = np.exp(g_t)[:, :, None] * S
    o = scale * np.einsum("hk,hkv->hv", q_t, S)
    read = np.einsum("hk,hkv->hv", k_t, S)
    u = beta_t[:, None] * (v_t - read) if delta else v_t
    return S + k_t[:, :, None] * u[:, None, :], o


def _step_transposed_read(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    S = np.exp(g_t)[:, :, None] * S
    if delta and S.shape[1] == S.shape[2]:
        read = np.einsum("hk,hvk->hv", k_t, S)
    else:
        read = np.einsum("hk,hkv->hv", k_t, S)
    u = beta_t[:, None] * (v_t - read) if delta else v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    return S, scale * np.einsum("hk,hkv->hv", q_t, S)


def _step_no_beta(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    S = np.exp(g_t)[:, :, None] * S
    u = (v_t - np.einsum("hk,hkv->hv", k_t, S)) if delta else v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    return S, scale * np.einsum("hk,hkv->hv", q_t, S)


def _step_plus_read(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    S = np.exp(g_t)[:, :, None] * S
    u = beta_t[:, None] * (v_t + np.einsum("hk,hkv->hv", k_t, S)) if delta else v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    return S, scale * np.einsum("hk,hkv->hv", q_t, S)


def _step_decay_value_axis(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    if S.shape[1] == S.shape[2]:
        S = np.exp(g_t)[:, None, :] * S
    else:
        S = np.exp(g_t)[:, :, None] * S
    u = beta_t[:, None] * (v_t - np.einsum("hk,hkv->hv", k_t, S)) if delta else v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    return S, scale * np.einsum("hk,hkv->hv", q_t, S)


def _step_no_scale(S, q_t, k_t, v_t, g_t, beta_t, scale, delta):
    S = np.exp(g_t)[:, :, None] * S
    u = beta_t[:, None] * (v_t - np.einsum("hk,hkv->hv", k_t, S)) if delta else v_t
    S = S + k_t[:, :, None] * u[:, None, :]
    return S, np.einsum("hk,hkv->hv", q_t, S)


def _gate_no_exp(a, dt_bias, A_log):
    return -np.asarray(A_log)[:, None] * ko.softplus(np.asarray(a) + np.asarray(dt_bias))


def _gate_no_bias(a, dt_bias, A_log):
    return -np.exp(np.asarray(A_log))[:, None] * ko.softplus(np.asarray(a))


def _l2_no_eps(x):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def _sigmoid_wrong(x):
    return 1.0 / (1.0 + np.exp(np.asarray(x, np.float64)))


def _fs_wrong_sign(L, R):
    X = np.array(np.asarray(R, np.float64))
    for i in range(L.shape[-1]):
        for j in range(i):
            X[..., i, :] += L[..., i, j, None] * X[..., j, :]
    return X


def _neumann_short(L):
    n = L.shape[-1]
    eye = np.broadcast_to(np.eye(n), L.shape)
    X = -np.asarray(L)
    X2 = X @ X
    return (eye + X) @ (eye + X2) @ (eye + X2 @ X2)


def _cm_exclusive_cumsum(q, k, g, beta, scale):
    g = np.asarray(g, np.float64)
    shifted = np.concatenate([np.zeros_like(g[:1]), g[:-1]], axis=0)
    return _orig_chunk_matrices(q, k, shifted, beta, scale)


def _cm_diag_in_L(q, k, g, beta, scale):
    m = _orig_chunk_matrices(q, k, g, beta, scale)
    kk = np.einsum("ihc,ihc->hi", np.asarray(k), np.asarray(k))
    n = m["L"].shape[-1]
    m["L"] = m["L"] + np.asarray(beta).T[:, :, None] * kk[:, :, None] * np.eye(n)[None]
    return m


def _cm_no_beta(q, k, g, beta, scale):
    return _orig_chunk_matrices(q, k, g, np.ones_like(np.asarray(beta, np.float64)), scale)


_orig_chunk_matrices = ko.chunk_matrices
_orig_recurrent_pool = ko.kda_recurrent_pool


def _conv_taps_reversed(x, conv_state, weight, bias):
    return ko_conv_orig(x, conv_state, np.asarray(weight)[:, ::-1], bias)


def _conv_no_shift(x, conv_state, weight, bias):
    y, _ = ko_conv_orig(x, conv_state, weight, bias)
    return y, np.asarray(conv_state, np.float64)


def _silu_plain_sigmoid(x):
    return ko.sigmoid(x)


ko_conv_orig = ko.causal_conv1d_update
_orig_decode_conv = ko.kda_decode_conv
_orig_chunk_start_states = ko.chunk_start_states


def _cs_after_not_before(q, k, v, g, beta, scale, C, h0=None, delta=True):
    snaps = _orig_chunk_start_states(q, k, v, g, beta, scale, C, h0=h0, delta=delta)
    _, hT = ko.kda_recurrent(q, k, v, g, beta, scale, h0=h0, delta=delta)
    return np.concatenate([snaps[1:], hT[None]], axis=0)


def _dc_conv_on_pads(mixed_qkv, conv_state, conv_weight, conv_bias, *args, **kw):
    o, pool, cs = _orig_decode_conv(mixed_qkv, conv_state, conv_weight, conv_bias, *args, **kw)
    idx = np.asarray(args[5])
    cs = np.array(cs)
    for row in np.nonzero(idx < 0)[0]:
        _, cs[(row + 1) % cs.shape[0]] = ko.causal_conv1d_update(mixed_qkv[row], cs[(row + 1) % cs.shape[0]],
                                                                 conv_weight, conv_bias)
    return o, pool, cs


def _dc_no_activation(mixed_qkv, conv_state, conv_weight, conv_bias, *args, **kw):
    saved = ko.silu
    ko.silu = lambda x: np.asarray(x, np.float64)
    try:
        return _orig_decode_conv(mixed_qkv, conv_state, conv_weight, conv_bias, *args, **kw)
    finally:
        ko.silu = saved


def _rms_no_weight(x, weight, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rms_sum_not_mean(x, weight, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * np.asarray(weight)


def _rms_eps_outside(x, weight, eps):
    x = np.asarray(x, np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * np.asarray(weight)


def _hg_first_channel_only(g_head, K):
    g = np.asarray(g_head, np.float64)
    out = np.zeros(g.shape + (K,))
    out[..., 0] = g
    return out


def _hg_exp_twice(g_head, K):
    return np.repeat(np.exp(np.asarray(g_head, np.float64))[..., None] - 1.0, K, axis=-1)


def _rp_reversed_tokens(q, k, v, a, b, *args, **kw):
    return _orig_recurrent_pool(q[:, ::-1], k[:, ::-1], v[:, ::-1], a[:, ::-1], b[:, ::-1], *args, **kw)


def _rp_group_by_modulo(q, k, v, a, b, A_log, dt_bias, state_pool, indices, *, scale, l2norm_qk=True):
    H, HV = q.shape[2], v.shape[2]
    qm = np.asarray(q)[:, :, np.arange(HV) % H]
    km = np.asarray(k)[:, :, np.arange(HV) % H]
    return _orig_recurrent_pool(qm, km, v, a, b, A_log, dt_bias, state_pool, indices, scale=scale,
                                l2norm_qk=l2norm_qk)


def _rp_state_not_carried(q, k, v, a, b, A_log, dt_bias, state_pool, indices, *, scale, l2norm_qk=True):
    outs = []
    for t in range(np.asarray(q).shape[1]):
        ot, newp = _orig_recurrent_pool(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], a[:, t:t + 1], b[:, t:t + 1],
                                        A_log, dt_bias, state_pool, indices, scale=scale, l2norm_qk=l2norm_qk)
        outs.append(ot)
    return np.concatenate(outs, axis=1), newp


MUTANTS = [
    ("_token_step", _step_decay_after_write),
    ("_token_step", _step_read_before_write),
    ("_token_step", _step_transposed_read),
    ("_token_step", _step_no_beta),
    ("_token_step", _step_plus_read),
    ("_token_step", _step_decay_value_axis),
    ("_token_step", _step_no_scale),
    ("kda_gate", _gate_no_exp),
    ("kda_gate", _gate_no_bias),
    ("l2_normalize", _l2_no_eps),
    ("sigmoid", _sigmoid_wrong),
    ("forward_substitution", _fs_wrong_sign),
    ("neumann_inverse", _neumann_short),
    ("chunk_matrices", _cm_exclusive_cumsum),
    ("chunk_matrices", _cm_diag_in_L),
    ("chunk_matrices", _cm_no_beta),
    ("kda_recurrent_pool", _rp_reversed_tokens),
    ("kda_recurrent_pool", _rp_group_by_modulo),
    ("kda_recurrent_pool", _rp_state_not_carried),
    ("head_gate_to_channels", _hg_first_channel_only),
    ("head_gate_to_channels", _hg_exp_twice),
    ("head_rmsnorm", _rms_no_weight),
    ("head_rmsnorm", _rms_sum_not_mean),
    ("head_rmsnorm", _rms_eps_outside),
    ("causal_conv1d_update", _conv_taps_reversed),
    ("causal_conv1d_update", _conv_no_shift),
    ("silu", _silu_plain_sigmoid),
    ("kda_decode_conv", _dc_conv_on_pads),
    ("kda_decode_conv", _dc_no_activation),
    ("chunk_start_states", _cs_after_not_before),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_mutants_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(ko, name, mutant)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutant.__name__} in {name} went unnoticed by every pin"
