"""Pins of the chunk-form backward restatement (oracle/chunk_backward.py)
against the per-token backward oracle (itself pinned to finite differences
in test_oracle_backward_pins.py): every gradient for the scalar and the
per-dim gate, chunk sizes 1, 5, 16 and 64 (ragged last chunks), packed
sequences, an output scale and a final-state gradient.  Plus a planted
mistake in the restatement that the comparison catches."""
import numpy as np
import pytest

import oracle
from oracle import chunk_backward as cb


def rand_problem(rng, T, H, dk, dv, gate):
    def unit(shape):
        x = rng.standard_normal(shape)
        return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)

    q = unit((1, T, H, dk))
    k = unit((1, T, H, dk))
    v = rng.standard_normal((1, T, H, dv)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((1, T, H))))).astype(np.float32)
    gshape = (1, T, H) if gate == "gdn" else (1, T, H, dk)
    g = (-np.log1p(np.exp(-(2.0 + rng.standard_normal(gshape))))).astype(np.float32)
    return dict(q=q, k=k, v=v, beta=beta, g=g)


def reference(p, do, dht, cu, scale):
    return oracle.Problem(**p, cu_seqlens=cu, scale=scale).backward(do, dht=dht, nthreads=1)


@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("C", [1, 5, 16, 64])
def test_chunk_backward_matches_per_token_backward(gate, C):
    rng = np.random.default_rng(101 + C + (0 if gate == "gdn" else 7))
    T, H, dk, dv = 150, 2, 8, 6
    cu = [0, 37, 101, 150]
    scale = 0.6
    p = rand_problem(rng, T, H, dk, dv, gate)
    do = rng.standard_normal((1, T, H, dv)).astype(np.float32)
    dht = rng.standard_normal((3, H, dk, dv))
    ref = reference(p, do, dht, cu, scale)
    got = cb.chunked_backward(p["q"], p["k"], p["v"], p["beta"], p["g"], do, dht=dht, C=C, scale=scale,
                              cu_seqlens=cu)
    for name in ("dq", "dk", "dv", "dbeta", "dg"):
        r, x = ref[name], got[name]
        err = np.abs(x - r).max() / max(np.abs(r).max(), 1e-30)
        assert err < 1e-9, (name, err)


def test_chunk_backward_without_final_state_gradient_and_unpacked_rows():
    rng = np.random.default_rng(211)
    T, H, dk, dv = 70, 1, 5, 4
    p = rand_problem(rng, T, H, dk, dv, "gdn")
    p = {key: np.concatenate([x, x[:, ::-1]], axis=0) for key, x in p.items()}   # B = 2 rows
    do = rng.standard_normal((2, T, H, dv)).astype(np.float32)
    ref = oracle.Problem(**p).backward(do, nthreads=1)
    got = cb.chunked_backward(p["q"], p["k"], p["v"], p["beta"], p["g"], do, C=16)
    for name in ("dq", "dk", "dv", "dbeta", "dg"):
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-12, err_msg=name)


def test_planted_mistake_is_caught(monkeypatch):
    """Dropping the decay of the carried state gradient (Diag(gC) dS') must
    break the agreement (the comparison is not vacuous)."""
    rng = np.random.default_rng(307)
    T, H, dk, dv = 40, 1, 4, 3
    p = rand_problem(rng, T, H, dk, dv, "gdn")
    do = rng.standard_normal((1, T, H, dv)).astype(np.float32)
    ref = reference(p, do, None, None, 1.0)
    real = cb._chunk_backward

    def broken(Q, K, V, beta, G, S, c, dO, dSn, scale):
        out = list(real(Q, K, V, beta, G, S, c, dO, dSn, scale))
        out[5] = out[5] - (c["gC"][:, None] - 1.0) * dSn   # dS with dS' not decayed
        return tuple(out)

    monkeypatch.setattr(cb, "_chunk_backward", broken)
    got = cb.chunked_backward(p["q"], p["k"], p["v"], p["beta"], p["g"], do, C=8)
    worst = max(np.abs(got[n] - ref[n]).max() / np.abs(ref[n]).max() for n in ("dq", "dk", "dv", "dbeta", "dg"))
    assert worst > 1e-3
