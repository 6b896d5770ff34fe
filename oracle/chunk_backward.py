"""fp64 restatement of the backward in chunk (WY) form.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: the tests call it;
the CUDA library shares nothing with it.

Source: the article "flash-linear-attention 上下文并行CP 从 CP2TP、Ring CP 到
True CP 的设计取舍与源码实现" ([FLA-CP]).  §2.2 gives the chunk form of the
forward that ``oracle.c``'s ``chunk_pass`` restates; §4 lists the backward's
flow (the chunk-level state-gradient chain and the per-chunk input
gradients through the WY inverse).  The pages print no backward formulas, so
this module is the plain reverse-mode derivative of the chunk equations,
chunk by chunk from the last, written out (per-dim gates G, n x dk, cover
both gate kinds: a scalar gate repeats across the key dims):

  forward of one chunk (natural-log gates, cumulative inside the chunk)
    E = exp(G), Qg = Q*E, Kg = K*E, Kn = K*exp(-G), KgC = K*exp(G_C - G),
    gC = exp(G_C),  G_C = last row of G
    A = strict_lower(diag(beta) Kg Kn^T),  T = (I + A)^-1
    P = lower_incl(Qg Kn^T)
    W = T diag(beta) Kg,  U = T diag(beta) V,  Delta = U - W S
    O = scale (Qg S + P Delta),  S' = Diag(gC) S + KgC^T Delta

  backward, given dO and dS' (the state gradient after the chunk)
    dDelta = P^T dO~ + KgC dS'                   (dO~ = scale dO)
    dS     = Diag(gC) dS' + Qg^T dO~ - W^T dDelta
    dP = lower_incl(dO~ Delta^T):  dQg = dO~ S^T + dP Kn,  dKn = dP^T Qg
    dW = -dDelta S^T,  dU = dDelta,  dKgC = Delta dS'^T,  dgC = rowsum(dS' * S)
    through W and U:  dKg = beta * (T^T dW),  dV = beta * (T^T dU),
                      dbeta = rowsum((T^T dW) * Kg) + rowsum((T^T dU) * V),
                      dT = dW (diag(beta) Kg)^T + dU (diag(beta) V)^T
    through T:        dA = strict_lower(-T^T dT T^T)
    through A:        Y = Kg Kn^T,  dbeta += rowsum(dA * Y),
                      dKg += (beta * dA) Kn,  dKn += (beta * dA)^T Kg
    to Q, K, G:       dQ = dQg * E,  dK = dKg * E + dKn * exp(-G) + dKgC * exp(G_C - G)
                      dG = dQg * Qg + dKg * Kg - dKn * Kn - dKgC * KgC,
                      dG_C += colsum(dKgC * KgC) + dgC * gC
    the per-token gate gradient is the reverse cumulative sum of dG inside the
    chunk (summed over key dims for a scalar gate); dS carries to the
    previous chunk.

The per-token backward in ``oracle.c`` (pinned by finite differences) is the
definition; this restatement is pinned against it in
``tests/test_oracle_chunk_backward_pins.py`` at several chunk sizes.
"""
from __future__ import annotations

import numpy as np


def _chunk_forward(Q, K, V, beta, G, S):
    """One chunk's intermediates (all fp64); G: n x dk cumulative log gates."""
    n = K.shape[0]
    E, En = np.exp(G), np.exp(-G)
    GC = G[-1]
    gC = np.exp(GC)
    Qg, Kg, Kn = Q * E, K * E, K * En
    KgC = K * np.exp(GC[None, :] - G)
    A = np.tril(beta[:, None] * (Kg @ Kn.T), -1)
    T = np.linalg.inv(np.eye(n) + A)
    P = np.tril(Qg @ Kn.T)
    W = T @ (beta[:, None] * Kg)
    U = T @ (beta[:, None] * V)
    D = U - W @ S
    return dict(E=E, En=En, GC=GC, gC=gC, Qg=Qg, Kg=Kg, Kn=Kn, KgC=KgC, T=T, P=P, W=W, D=D)


def _chunk_backward(Q, K, V, beta, G, S, c, dO, dSn, scale):
    """Gradients of one chunk; returns (dQ, dK, dV, dbeta, dG, dS)."""
    dOs = scale * dO
    T, P, W, D = c["T"], c["P"], c["W"], c["D"]
    Qg, Kg, Kn, KgC = c["Qg"], c["Kg"], c["Kn"], c["KgC"]
    dD = P.T @ dOs + KgC @ dSn
    dS = c["gC"][:, None] * dSn + Qg.T @ dOs - W.T @ dD
    dP = np.tril(dOs @ D.T)
    dQg = dOs @ S.T + dP @ Kn
    dKn = dP.T @ Qg
    dW = -dD @ S.T
    dU = dD
    dKgC = D @ dSn.T
    dgC = np.sum(dSn * S, axis=1)
    TtW, TtU = T.T @ dW, T.T @ dU
    dKg = beta[:, None] * TtW
    dV = beta[:, None] * TtU
    dbeta = np.sum(TtW * Kg, axis=1) + np.sum(TtU * V, axis=1)
    dT = dW @ (beta[:, None] * Kg).T + dU @ (beta[:, None] * V).T
    dA = np.tril(-(T.T @ dT @ T.T), -1)
    Y = Kg @ Kn.T
    dbeta = dbeta + np.sum(dA * Y, axis=1)
    bdA = beta[:, None] * dA
    dKg = dKg + bdA @ Kn
    dKn = dKn + bdA.T @ Kg
    E, En = c["E"], c["En"]
    dQ = dQg * E
    dK = dKg * E + dKn * En + dKgC * np.exp(c["GC"][None, :] - G)
    dG = dQg * Qg + dKg * Kg - dKn * Kn - dKgC * KgC
    dG[-1] += np.sum(dKgC * KgC, axis=0) + dgC * c["gC"]
    return dQ, dK, dV, dbeta, dG, dS


def chunked_backward(q, k, v, beta, g, do, dht=None, C=64, scale=1.0, cu_seqlens=None):
    """Chunk-form gradients of sum <do, o> + sum <dht, S_final>, zero initial state.

    q, k: [B, T, H, dk]; v, do: [B, T, H, dv]; beta: [B, T, H]; g: [B, T, H]
    (scalar gate) or [B, T, H, dk] (per-dim), natural-log; dht: [N, H, dk, dv]
    or None.  With ``cu_seqlens`` the batch is packed (B == 1).  Returns a dict
    of fp64 dq, dk, dv, dbeta, dg in the inputs' shapes.
    """
    as64 = lambda x: np.asarray(x, dtype=np.float64)
    q, k, v, beta, g, do = (as64(x) for x in (q, k, v, beta, g, do))
    B, Tn, H, dk = k.shape
    dv = v.shape[3]
    scalar = g.ndim == 3
    if cu_seqlens is None:
        ranges = [(b, 0, Tn) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens]
        ranges = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dbeta=np.zeros_like(beta),
               dg=np.zeros_like(g))
    for n, (b, s, e) in enumerate(ranges):
        for h in range(H):
            starts = list(range(s, e, C))
            # forward: the state at each chunk start and the chunk intermediates
            S = np.zeros((dk, dv))
            saved = []
            for c0 in starts:
                c1 = min(c0 + C, e)
                gg = g[b, c0:c1, h]
                gd = np.repeat(gg[:, None], dk, axis=1) if scalar else gg
                G = np.cumsum(gd, axis=0)
                c = _chunk_forward(q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h], beta[b, c0:c1, h], G, S)
                saved.append((c0, c1, G, S, c))
                S = c["gC"][:, None] * S + c["KgC"].T @ c["D"]
            # backward from the final state's gradient
            dS = np.zeros((dk, dv)) if dht is None else as64(dht)[n, h].copy()
            for c0, c1, G, S0, c in reversed(saved):
                dQ, dK, dV, dB, dG, dS = _chunk_backward(q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h],
                                                         beta[b, c0:c1, h], G, S0, c, do[b, c0:c1, h], dS, scale)
                out["dq"][b, c0:c1, h] = dQ
                out["dk"][b, c0:c1, h] = dK
                out["dv"][b, c0:c1, h] = dV
                out["dbeta"][b, c0:c1, h] = dB
                dg_tok = np.cumsum(dG[::-1], axis=0)[::-1]
                out["dg"][b, c0:c1, h] = dg_tok.sum(axis=1) if scalar else dg_tok
    return out
