"""Pins of the backward oracle (the reverse of the per-token scan) to
central finite differences of the forward oracle, on tiny problems in fp64
arithmetic: every gradient (q, k, v, beta, gate) for the scalar and the
per-dim gate, packed sequences, an output scale and a final-state
gradient, with and without grouped query heads.  Plus the scalar gate as
the per-dim gate constant across dims, and grouped query heads as the same
problem with every state input repeated per group (gradients of the copies
summed)."""
import numpy as np
import pytest

import oracle


def rand_problem(rng, T, H, dk, dv, gate, G=1):
    def unit(shape):
        x = rng.standard_normal(shape)
        return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)

    q = unit((1, T, H * G, dk))
    k = unit((1, T, H, dk))
    v = rng.standard_normal((1, T, H, dv)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((1, T, H))))).astype(np.float32)
    gshape = (1, T, H) if gate == "gdn" else (1, T, H, dk)
    g = (-np.log1p(np.exp(-(1.0 + rng.standard_normal(gshape))))).astype(np.float32)
    return dict(q=q, k=k, v=v, beta=beta, g=g)


def loss(p, cu, scale, W_o, W_s):
    o, ht = oracle.Problem(**p, cu_seqlens=cu, scale=scale).scan()
    return float((o * W_o).sum() + (ht * W_s).sum())


@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_backward_matches_finite_differences(gate, G):
    rng = np.random.default_rng((31 if gate == "gdn" else 32) + 10 * (G - 1))
    T, H, dk, dv = 7, 2, 3, 2
    cu = [0, 3, 7]
    scale = 0.7
    p = rand_problem(rng, T, H, dk, dv, gate, G)
    W_o = rng.standard_normal((1, T, H * G, dv)).astype(np.float32)
    W_s = rng.standard_normal((2, H, dk, dv))
    grads = oracle.Problem(**p, cu_seqlens=cu, scale=scale).backward(W_o, dht=W_s)
    names = dict(q="dq", k="dk", v="dv", beta="dbeta", g="dg")
    for key, gname in names.items():
        x = p[key]
        fd = np.zeros(x.shape)
        for idx in np.ndindex(x.shape):
            eps = 1e-3 * max(1.0, abs(float(x[idx])))
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            h = float(xp[idx]) - float(xm[idx])   # the step the fp32 inputs actually took
            fd[idx] = (loss(dict(p, **{key: xp}), cu, scale, W_o, W_s) -
                       loss(dict(p, **{key: xm}), cu, scale, W_o, W_s)) / h
        np.testing.assert_allclose(grads[gname], fd, rtol=2e-4, atol=2e-6, err_msg=gname)


def test_scalar_gate_is_constant_per_dim_gate():
    rng = np.random.default_rng(33)
    T, H, dk, dv = 20, 2, 4, 3
    p = rand_problem(rng, T, H, dk, dv, "gdn")
    pk = dict(p, g=np.repeat(p["g"][..., None], dk, axis=-1))
    do = rng.standard_normal((1, T, H, dv)).astype(np.float32)
    a = oracle.Problem(**p).backward(do)
    b = oracle.Problem(**pk).backward(do)
    for key in ("dq", "dk", "dv", "dbeta"):
        np.testing.assert_allclose(a[key], b[key], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a["dg"], b["dg"].sum(-1), rtol=1e-12, atol=1e-14)


def test_long_sequence_crosses_checkpoints():
    """T = 150: the states are recomputed from checkpoints every 64 tokens;
    finite differences at tokens next to the checkpoints (63, 64, 65, 128)
    and at both ends."""
    rng = np.random.default_rng(34)
    T, H, dk, dv = 150, 1, 4, 3
    p = rand_problem(rng, T, H, dk, dv, "kda")
    W_o = rng.standard_normal((1, T, H, dv)).astype(np.float32)
    W_s = rng.standard_normal((1, H, dk, dv))
    grads = oracle.Problem(**p).backward(W_o, dht=W_s)
    for t in (0, 63, 64, 65, 128, 149):
        for key, gname, idx in (("k", "dk", (0, t, 0, 1)), ("v", "dv", (0, t, 0, 2)), ("beta", "dbeta", (0, t, 0)),
                                ("g", "dg", (0, t, 0, 3)), ("q", "dq", (0, t, 0, 0))):
            x = p[key]
            eps = 1e-3 * max(1.0, abs(float(x[idx])))
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            h = float(xp[idx]) - float(xm[idx])
            fd = (loss(dict(p, **{key: xp}), None, 1.0, W_o, W_s) - loss(dict(p, **{key: xm}), None, 1.0, W_o, W_s)) / h
            np.testing.assert_allclose(grads[gname][idx], fd, rtol=2e-4, atol=2e-6, err_msg=f"{gname} at {t}")


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_grouped_query_heads_equal_repeated_state_inputs(gate):
    """G query heads per state: the same loss as a problem with k, v, beta and
    the gate repeated G times (one state per query head, each an identical
    copy), so dq is the same and each state gradient is the sum over its
    group of the copies' gradients; the final-state gradient of a state goes
    to its first copy."""
    rng = np.random.default_rng(35)
    G, T, H, dk, dv = 3, 19, 2, 4, 3
    cu = [0, 8, 19]
    p = rand_problem(rng, T, H, dk, dv, gate, G)
    do = rng.standard_normal((1, T, H * G, dv)).astype(np.float32)
    dht = rng.standard_normal((2, H, dk, dv))
    a = oracle.Problem(**p, cu_seqlens=cu, scale=0.6).backward(do, dht=dht)
    rep = dict(p, **{key: np.repeat(p[key], G, axis=2) for key in ("k", "v", "beta", "g")})
    dht_rep = np.zeros((2, H * G, dk, dv))
    dht_rep[:, ::G] = dht
    b = oracle.Problem(**rep, cu_seqlens=cu, scale=0.6).backward(do, dht=dht_rep)
    np.testing.assert_allclose(a["dq"], b["dq"], rtol=1e-12, atol=1e-14)
    for key in ("dk", "dv", "dbeta", "dg"):
        y = b[key]
        summed = y.reshape(y.shape[:2] + (H, G) + y.shape[3:]).sum(axis=3)
        np.testing.assert_allclose(a[key], summed, rtol=1e-11, atol=1e-13, err_msg=key)
