"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the article or plain
mathematics fixes: brute-force explicit matrix products on tiny inputs,
closed forms (EMA, orthonormal-key linear attention, delta overwrite,
Householder orthogonality), gate-free and beta-free special cases, the
segmented == whole-sequence invariant (hyper-parallel issue #7, KDA
initial_state comment: H0 -> ... -> HT, segment 2 starting from segment 1's
state), and the chunk form of the article "flash-linear-attention 上下文并行CP
..." (§2.2) against the per-token definition.  Chosen so that a dropped term,
a wrong sign, a transposed operand or a wrong merge order fails at least one.
"""
import numpy as np
import pytest

import oracle


def rand_problem(rng, B=1, T=12, H=2, dk=8, dv=6, gate="gdn", cu=None, gmu=2.0, gs=1.0):
    def unit(shape):
        x = rng.standard_normal(shape).astype(np.float32)
        return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)

    q = unit((B, T, H, dk))
    k = unit((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, T, H))))).astype(np.float32)
    gshape = (B, T, H) if gate == "gdn" else (B, T, H, dk)
    z = gmu + gs * rng.standard_normal(gshape)
    g = (-np.log1p(np.exp(-z))).astype(np.float32)
    return dict(q=q, k=k, v=v, beta=beta, g=g, cu_seqlens=cu)


def alphas(p, t, h, dk):
    g = p["g"][0, t, h].astype(np.float64)
    return np.exp(g) * np.ones(dk) if np.ndim(g) == 0 else np.exp(g)


def brute_force_single(p, h, t0, t1, S0):
    """Explicit matrices: S_t = T_t S_{t-1} + b_t k_t v_t^T with
    T_t = (I - b k k^T) Diag(alpha), unrolled as a sum over tokens of
    (prod_{s>t} T_s) b_t k_t v_t^T plus (prod T) S0; outputs S_t^T q_t."""
    dk = p["k"].shape[3]
    Ts, adds, outs = [], [], []
    for t in range(t0, t1):
        k = p["k"][0, t, h].astype(np.float64)
        b = float(p["beta"][0, t, h])
        Tt = (np.eye(dk) - b * np.outer(k, k)) @ np.diag(alphas(p, t, h, dk))
        Ts.append(Tt)
        adds.append(b * np.outer(k, p["v"][0, t, h].astype(np.float64)))
    for i in range(len(Ts)):
        # S_i = (T_i ... T_0) S0 + sum_{j<=i} (T_i ... T_{j+1}) add_j
        P = np.eye(dk)
        S = np.zeros_like(S0)
        for j in range(i, -1, -1):
            S = S + P @ adds[j]
            P = P @ Ts[j]
        S = S + P @ S0
        outs.append(S.T @ p["q"][0, t0 + i, h].astype(np.float64))
    return np.array(outs), (S if Ts else S0)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_brute_force_tiny(gate):
    rng = np.random.default_rng(1)
    p = rand_problem(rng, T=13, H=2, dk=5, dv=3, gate=gate)
    o, ht = oracle.Problem(**p).scan()
    for h in range(2):
        ob, Sb = brute_force_single(p, h, 0, 13, np.zeros((5, 3)))
        np.testing.assert_allclose(o[0, :, h], ob, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(ht[0, h], Sb, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_brute_force_segment_quantities(gate):
    """S_ext, M of a trailing fragment as explicit products; S_init by the
    article's merge loop S <- M_j S + S_ext,j, over tiny packed sequences."""
    rng = np.random.default_rng(2)
    lengths = [3, 10, 3]          # total 16, R = 4 -> L = 4; sequence 1 spans segments 0..3
    cu = np.cumsum([0] + lengths)
    p = rand_problem(rng, T=16, H=1, dk=4, dv=3, gate=gate, cu=cu)
    out = oracle.Problem(**p).segmented(4)
    dk = 4
    # segment 0: trailing fragment [3, 4) of sequence 1; segment 1: [4, 8); segment 2: [8, 12)
    for r, (f0, f1) in enumerate([(3, 4), (4, 8), (8, 12)]):
        M = np.eye(dk)
        S = np.zeros((dk, 3))
        for t in range(f0, f1):
            k = p["k"][0, t, 0].astype(np.float64)
            b = float(p["beta"][0, t, 0])
            Tt = (np.eye(dk) - b * np.outer(k, k)) @ np.diag(alphas(p, t, 0, dk))
            M = Tt @ M
            S = Tt @ S + b * np.outer(k, p["v"][0, t, 0].astype(np.float64))
        np.testing.assert_allclose(out["M"][r, 0, 0], M, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["S_ext"][r, 0, 0], S, rtol=1e-12, atol=1e-14)
    # segment 3 ends where its last sequence ends: nothing crosses
    assert not out["S_ext"][3].any() and not out["M"][3].any()
    # the merge: segment 1 needs only segment 0; segment 3 needs 0, 1, 2
    E, Mm = out["S_ext"][:, 0, 0], out["M"][:, 0, 0]
    np.testing.assert_allclose(out["S_init"][1, 0, 0], E[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out["S_init"][2, 0, 0], Mm[1] @ E[0] + E[1], rtol=1e-12, atol=1e-14)
    s3 = Mm[2] @ (Mm[1] @ E[0] + E[1]) + E[2]
    np.testing.assert_allclose(out["S_init"][3, 0, 0], s3, rtol=1e-12, atol=1e-14)
    assert not out["S_init"][0].any()


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_ema_closed_form(gate):
    """k_t = e_0, alpha_t = a (per dim a_d for KDA), beta_t = b:
    row 0 of S follows s_t = a_0 (1 - b) s_{t-1} + b v_t, other rows stay 0,
    o_t = (q_t . e_0) s_t."""
    T, dk, dv = 40, 6, 4
    rng = np.random.default_rng(3)
    k = np.zeros((1, T, 1, dk), np.float32)
    k[..., 0] = 1.0
    q = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, dv)).astype(np.float32)
    beta = np.full((1, T, 1), 0.375, np.float32)
    if gate == "gdn":
        g = np.full((1, T, 1), np.log(0.875), np.float32)
        a0 = float(np.exp(np.float64(g[0, 0, 0])))
    else:
        g = np.log(np.linspace(0.5, 0.95, dk, dtype=np.float32))[None, None, None, :].repeat(T, 1)
        g = np.ascontiguousarray(g, np.float32)
        a0 = float(np.exp(np.float64(g[0, 0, 0, 0])))
    o, ht = oracle.Problem(q, k, v, beta, g).scan()
    s = np.zeros(dv)
    b = 0.375
    for t in range(T):
        s = a0 * (1 - b) * s + b * v[0, t, 0].astype(np.float64)
        np.testing.assert_allclose(o[0, t, 0], float(q[0, t, 0, 0]) * s, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ht[0, 0, 0], s, rtol=1e-12)
    assert not ht[0, 0, 1:].any()


def test_orthonormal_keys_are_linear_attention():
    """alpha = 1 and k_t = e_t (t < dk): every write hits a fresh row, so
    o_t = sum_{tau <= t} beta_tau q_t[tau] v_tau (plain causal linear attention)."""
    T = dk = 8
    dv = 5
    rng = np.random.default_rng(4)
    k = np.eye(dk, dtype=np.float32)[None, :, None, :]
    q = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, dv)).astype(np.float32)
    beta = rng.uniform(0.1, 0.9, (1, T, 1)).astype(np.float32)
    g = np.zeros((1, T, 1), np.float32)
    o, _ = oracle.Problem(q, k, v, beta, g).scan()
    Q, V, Bt = q[0, :, 0].astype(np.float64), v[0, :, 0].astype(np.float64), beta[0, :, 0].astype(np.float64)
    ref = np.tril(Q) * Bt[None, :] @ V       # (q_t[tau] masked tau <= t) * beta_tau @ v_tau
    np.testing.assert_allclose(o[0, :, 0], ref, rtol=1e-12, atol=1e-14)


def test_delta_rule_overwrites():
    """beta = 1, alpha = 1, one repeated unit key e: the update replaces the
    value stored under e, so S_T = e v_T^T regardless of earlier writes."""
    T, dk, dv = 5, 4, 3
    rng = np.random.default_rng(5)
    k = np.zeros((1, T, 1, dk), np.float32)
    k[..., 2] = 1.0
    v = rng.standard_normal((1, T, 1, dv)).astype(np.float32)
    q = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    o, ht = oracle.Problem(q, k, v, np.ones((1, T, 1), np.float32), np.zeros((1, T, 1), np.float32)).scan()
    ref = np.zeros((dk, dv))
    ref[2] = v[0, -1, 0]
    np.testing.assert_allclose(ht[0, 0], ref, atol=1e-15)
    np.testing.assert_allclose(o[0, :, 0], q[0, :, 0, 2:3].astype(np.float64) * v[0, :, 0], atol=1e-15)


def test_householder_chain_is_orthogonal():
    """beta = 2, alpha = 1: each per-token map I - 2 k k^T (exact unit k) is a
    reflection, so the chained transfer matrix M is orthogonal with
    det = (-1)^(tokens), and with v = 0 the state norm is preserved."""
    T, dk, dv, R = 24, 8, 3, 2
    rng = np.random.default_rng(6)
    k = np.zeros((1, T, 1, dk), np.float32)
    for t in range(T):
        idx = rng.choice(dk, 4, replace=False)
        k[0, t, 0, idx] = rng.choice([-0.5, 0.5], 4)
    q = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    v = np.zeros((1, T, 1, dv), np.float32)
    out = oracle.Problem(q, k, v, np.full((1, T, 1), 2.0, np.float32),
                         np.zeros((1, T, 1), np.float32)).segmented(R)
    M = out["M"][0, 0, 0]
    np.testing.assert_allclose(M.T @ M, np.eye(dk), atol=1e-13)
    assert np.isclose(np.linalg.det(M), (-1.0) ** (T // R))
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, ht = oracle.Problem(q, k, v, np.full((1, T, 1), 2.0, np.float32),
                           np.zeros((1, T, 1), np.float32)).scan(h0=S0)
    assert np.isclose(np.linalg.norm(ht), np.linalg.norm(S0), rtol=1e-13)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_beta_zero(gate):
    """beta = 0: S_ext = 0 and M = Diag(prod of the fragment's alphas)."""
    rng = np.random.default_rng(7)
    p = rand_problem(rng, T=32, H=2, dk=6, dv=4, gate=gate)
    p["beta"][:] = 0
    out = oracle.Problem(**p).segmented(4)
    assert not out["S_ext"].any() and not out["o"].any()
    for r in range(3):
        for h in range(2):
            g = p["g"][0, r * 8:(r + 1) * 8, h].astype(np.float64)
            prod = np.exp(g.sum(0)) * np.ones(6) if gate == "gdn" else np.exp(g.sum(0))
            np.testing.assert_allclose(out["M"][r, 0, h], np.diag(prod), rtol=1e-13, atol=0)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_r1_is_the_plain_scan(gate):
    rng = np.random.default_rng(8)
    p = rand_problem(rng, B=2, T=20, H=3, dk=5, dv=4, gate=gate)
    P = oracle.Problem(**p)
    o, ht = P.scan()
    out = P.segmented(1)
    assert not out["S_init"].any() and not out["S_ext"].any() and not out["M"].any()
    np.testing.assert_array_equal(out["o"], o)
    np.testing.assert_array_equal(out["ht"], ht)


def serial_state_at(p, seq_start, h, t_end):
    """Serial-scan state of one head after global tokens [seq_start, t_end)."""
    sub = {}
    for name in ("q", "k", "v", "beta", "g"):
        a = p[name]
        sub[name] = np.ascontiguousarray(a.reshape((-1,) + a.shape[2:])[seq_start:t_end][None])
    sub["cu_seqlens"] = None
    _, ht = oracle.Problem(**sub).scan()
    return ht[0, h]


SEG_CASES = [
    # (B, T, lengths, R): fixed rows, and packed cut patterns scaled from the
    # article's §5.1 matrix: cut mid-sequence, aligned cut, one sequence over
    # three segments, many short sequences
    (2, 48, None, 4),
    (1, 48, [14, 19, 15], 2),
    (1, 48, [24, 24], 2),
    (1, 48, [33, 15], 4),
    (1, 48, [5, 7, 6, 9, 4, 11, 6], 2),
    (1, 64, [64], 8),
]


@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("case", SEG_CASES)
def test_segmented_equals_serial(gate, case):
    B, T, lengths, R = case
    rng = np.random.default_rng(9)
    cu = np.cumsum([0] + lengths) if lengths else None
    p = rand_problem(rng, B=B, T=T, H=2, dk=6, dv=5, gate=gate, cu=cu, gmu=3.0)
    P = oracle.Problem(**p)
    o, ht = P.scan()
    out = P.segmented(R)
    np.testing.assert_allclose(out["o"], o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["ht"], ht, rtol=1e-11, atol=1e-12)
    # S_init of every segment equals the serial state at the segment start
    L = T // R
    starts = [0] + list(np.cumsum(lengths)) if lengths else None
    for b in range(B):
        for r in range(R):
            t = (0 if lengths else b * T) + r * L
            if lengths:
                s = max(x for x in starts if x <= t)
                if s == t:
                    assert not out["S_init"][r, b].any()
                    continue
            else:
                s = b * T
                if r == 0:
                    assert not out["S_init"][r, b].any()
                    continue
            for h in range(2):
                ref = serial_state_at(p, s, h, t)
                np.testing.assert_allclose(out["S_init"][r, b, h], ref, rtol=1e-11, atol=1e-12)


def test_kda_constant_gate_is_gdn():
    rng = np.random.default_rng(10)
    p = rand_problem(rng, T=30, H=2, dk=6, dv=4, gate="gdn")
    pk = dict(p)
    pk["g"] = np.ascontiguousarray(np.repeat(p["g"][..., None], 6, axis=-1))
    a = oracle.Problem(**p).segmented(3)
    b = oracle.Problem(**pk).segmented(3)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunk_form_equals_serial(gate, C):
    """[FLA-CP] §2.2 chunk form (WY, forward substitution, Diag(gamma^C) decay)
    reproduces the per-token recurrence, including a partial last chunk."""
    rng = np.random.default_rng(11)
    lengths = [100, 37, 64]
    p = rand_problem(rng, T=201, H=2, dk=16, dv=8, gate=gate, cu=np.cumsum([0] + lengths), gmu=3.0)
    P = oracle.Problem(**p)
    o, ht = P.scan()
    oc, hc = P.chunked(C)
    np.testing.assert_allclose(oc, o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, ht, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_chunk_form_transfer_matrix(gate):
    """M chained as M <- M_[t] M with M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W
    equals the per-token product; S_ext likewise."""
    rng = np.random.default_rng(12)
    p = rand_problem(rng, T=160, H=2, dk=16, dv=8, gate=gate, gmu=3.0)
    P = oracle.Problem(**p)
    out = P.segmented(2)
    for h in range(2):
        S, M = P.chunked_pre(64, h, 0, 80)    # segment 0, three chunks (64 + 16)
        np.testing.assert_allclose(M, out["M"][0, 0, h], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(S, out["S_ext"][0, 0, h], rtol=1e-11, atol=1e-12)


def test_single_token_closed_form():
    """T = 1 from zero state: S_1 = beta k v^T, so o = scale * beta (k.q) v."""
    rng = np.random.default_rng(13)
    p = rand_problem(rng, T=1, H=3, dk=7, dv=5)
    o, _ = oracle.Problem(**p, scale=0.5).scan()
    for h in range(3):
        kq = float(np.dot(p["k"][0, 0, h].astype(np.float64), p["q"][0, 0, h].astype(np.float64)))
        ref = 0.5 * float(p["beta"][0, 0, h]) * kq * p["v"][0, 0, h].astype(np.float64)
        np.testing.assert_allclose(o[0, 0, h], ref, rtol=1e-13)


def test_gate_order_matters_only_for_per_dim_gates():
    rng = np.random.default_rng(14)
    p = rand_problem(rng, T=24, H=2, dk=6, dv=4, gate="gdn")
    a, _ = oracle.Problem(**p, order=0).scan()
    b, _ = oracle.Problem(**p, order=1).scan()
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    pk = rand_problem(rng, T=24, H=2, dk=6, dv=4, gate="kda", gmu=0.0)
    a, _ = oracle.Problem(**pk, order=0).scan()
    b, _ = oracle.Problem(**pk, order=1).scan()
    assert np.abs(a - b).max() > 1e-3 * np.abs(a).max()


def test_cut_rule():
    """[FLA-CP] §3.3: tokens per row must be >= R and divisible by R."""
    rng = np.random.default_rng(15)
    P = oracle.Problem(**rand_problem(rng, T=10, H=1, dk=4, dv=4))
    with pytest.raises(ValueError):
        P.segmented(4)
    with pytest.raises(ValueError):
        P.segmented(11)
    P.segmented(5)


def test_scale_is_linear():
    rng = np.random.default_rng(16)
    p = rand_problem(rng, T=9, H=1, dk=4, dv=3)
    a, _ = oracle.Problem(**p, scale=1.0).scan()
    b, _ = oracle.Problem(**p, scale=0.25).scan()
    np.testing.assert_allclose(b, 0.25 * a, rtol=1e-15)


# ---- grouped query heads ([FLA-CP] §5.1, GQA: Hq > H) --------------------
def _gqa_problem(rng, G, T=11, H=2, dk=5, dv=3, gate="gdn", cu=None, B=1):
    p = rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv, gate=gate, cu=cu)
    q = rng.standard_normal((B, T, H * G, dk)).astype(np.float32)
    p["q"] = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float32)
    return p


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_gqa_brute_force(gate):
    """Query head hq reads the state of head hq // G: explicit products per head."""
    G, H = 3, 2
    rng = np.random.default_rng(21)
    p = _gqa_problem(rng, G, H=H, gate=gate)
    o, ht = oracle.Problem(**p).scan()
    assert o.shape[2] == G * H and ht.shape[1] == H
    for hq in range(G * H):
        h = hq // G
        q2 = np.zeros_like(p["k"])
        q2[:, :, h] = p["q"][:, :, hq]
        ob, Sb = brute_force_single(dict(p, q=q2), h, 0, p["k"].shape[1], np.zeros((5, 3)))
        np.testing.assert_allclose(o[0, :, hq], ob, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(ht[0, h], Sb, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_gqa_equals_repeated_kv_heads(gate):
    """Grouping query heads is the same as repeating every other input per group."""
    G, H, R = 2, 3, 3
    rng = np.random.default_rng(22)
    p = _gqa_problem(rng, G, T=24, H=H, dk=6, dv=4, gate=gate, cu=[0, 5, 19, 24])
    rep = {k: np.repeat(p[k], G, axis=2) for k in ("k", "v", "beta", "g")}
    full = dict(p, **rep)
    a = oracle.Problem(**p).segmented(R)
    b = oracle.Problem(**full).segmented(R)
    np.testing.assert_array_equal(a["o"], b["o"])
    for key in ("ht", "S_ext", "M", "S_init"):
        x = a[key]
        y = b[key]
        hax = 1 if key == "ht" else 2
        np.testing.assert_array_equal(np.repeat(x, G, axis=hax), y)


def test_gqa_rejects_bad_grouping():
    rng = np.random.default_rng(23)
    p = _gqa_problem(rng, 1, H=2)
    p["q"] = p["q"][:, :, :1].repeat(3, axis=2)
    with pytest.raises(ValueError):
        oracle.Problem(**p)


# ---- token layouts ([FLA-CP] §3.2 zigzag) ---------------------------------
def test_zigzag_worked_example():
    """W = 2 ranks, 8 tokens: 4 parts of 2; rank 0 holds parts 0 and 3,
    rank 1 parts 1 and 2, each rank's input being [front; back]."""
    from oracle import layout
    np.testing.assert_array_equal(layout.zigzag_positions(8, 2), [0, 1, 6, 7, 2, 3, 4, 5])
    np.testing.assert_array_equal(layout.zigzag_positions(6, 3), [0, 5, 1, 4, 2, 3])
    np.testing.assert_array_equal(layout.zigzag_positions(10, 1), np.arange(10))


def test_zigzag_is_a_permutation_and_round_trips():
    from oracle import layout
    rng = np.random.default_rng(24)
    for total, W in [(64, 4), (96, 8), (4096, 16)]:
        pos = layout.zigzag_positions(total, W)
        assert sorted(pos.tolist()) == list(range(total))
        P = total // (2 * W)
        # every part is a run of P consecutive positions
        assert all((np.diff(pos[i * P:(i + 1) * P]) == 1).all() for i in range(2 * W))
        x = rng.standard_normal((2, total, 3))
        z = layout.to_zigzag(x, W)
        np.testing.assert_array_equal(z[:, np.argsort(pos)], x)
        np.testing.assert_array_equal(layout.from_zigzag(z, W), x)


def test_zigzag_cut_rule():
    """[FLA-CP] §3.3: zigzag needs total >= 2W and divisible by 2W."""
    from oracle import layout
    for total, W in [(6, 4), (10, 2), (3, 1)]:
        with pytest.raises(ValueError):
            layout.zigzag_positions(total, W)
