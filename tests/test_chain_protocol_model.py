"""A model of the forward chain kernel's synchronisation (csrc/tc_chain.cu),
checked by randomised interleavings on the CPU.

Each warp role (producer, MMA warp, mask warps, W/O epilogue warps, state
warps with the issuing lane) is written as the sequence of mbarrier waits,
arrivals, tensor-core products (asynchronous: their commits arrive when the
product completes, in issue order per issuing thread, in any order across
threads) and the shared-memory / TMEM accesses the kernel performs per
chunk, in the kernel's order.  A random scheduler runs them to completion
many times and fails on

* a deadlock (no role can proceed),
* a parity wait on a barrier that has already completed two phases past the
  one waited for (the hardware would report the wrong phase), and
* a data hazard: an access whose producer has not completed, or a write over
  data a reader has not consumed (each access states what must have
  happened before it).

Every role (and the products of each issuing thread) gets a random speed
for the whole schedule, so that one role lagging far behind the others is
explored as well as fair interleavings.

A mutation removes every wait on one barrier in the roles it names (for
the pre-process's WBFREE, both the MMA warp's and the W epilogue's: each
alone keeps the W tile from being rewritten while Delta reads it).

Models: the single-head forward (MODE_FWD) and its per-dim-gate form
(MODE_FWD_KDA: pre-gated Qg and P tiles with the stage), the forward of two
query heads per chain (MODE_FWD_G2: both heads' Q K^T in turn in the
columns W^T uses, both heads' outputs in one accumulator), and the
pre-process's S and M chains (MODE_PRE: a non-state warp issuing Delta and
P_S inside the state warps' named barrier), and the backward's
state-gradient chain (MODE_BWD).  The model is written from the kernel; it
does not run it.  Each model is also run with one wait removed, which the
checker must catch.
"""
import random
from collections import defaultdict

import pytest


class Protocol:
    """One random schedule of a set of role programs (generators of ops)."""

    def __init__(self, progs, counts, seed):
        self.rng = random.Random(seed)
        self.progs = progs
        self.counts = counts
        # each role (and each thread's products) runs at a random speed for
        # the whole schedule, so that one slow role lagging behind the rest
        # is explored as well as fair interleavings
        self.speed = {k: self.rng.choice([0.01, 0.1, 1.0]) for k in progs}

    def run(self):
        done, pend, acts, mdone = defaultdict(int), defaultdict(int), defaultdict(int), set()
        cur = {k: next(g) for k, g in self.progs.items()}
        inflight = defaultdict(list)
        barwait = set()

        def arrive(b):
            pend[b] += 1
            if pend[b] == self.counts.get(b, 1):
                pend[b] = 0
                done[b] += 1

        while True:
            runnable = []
            for k, op in cur.items():
                if op is None:
                    continue
                if op[0] == "wait":
                    b, j = op[1], op[2]
                    if done[b] >= j + 2:
                        return f"barrier {b} two phases ahead of {k} (wants {j}, {done[b]} done)"
                    if done[b] >= j + 1:
                        runnable.append(k)
                elif op[0] == "bar":
                    if k not in barwait:
                        runnable.append(k)
                else:
                    runnable.append(k)
            # the state warps' named barrier
            st = [k for k in cur if k.startswith("state") and cur[k] is not None]
            if st and all(cur[k][0] == "bar" and k in barwait for k in st):
                for k in st:
                    barwait.discard(k)
                    cur[k] = next(self.progs[k], None)
                continue
            choices = runnable + [("async", k) for k in inflight if inflight[k]]
            if not choices:
                if all(v is None for v in cur.values()):
                    return None
                return "deadlock: " + ", ".join(f"{k} at {v}" for k, v in cur.items() if v is not None)
            c = self.rng.choices(choices, [self.speed[x[1] if isinstance(x, tuple) else x] for x in choices])[0]
            if isinstance(c, tuple):   # the oldest product of that thread completes
                label, bars = inflight[c[1]].pop(0)
                mdone.add(label)
                for b in bars:
                    arrive(b)
                continue
            op = cur[c]
            if op[0] == "bar":
                barwait.add(c)
                continue
            if op[0] == "arrive":
                arrive(op[1])
            elif op[0] == "mma":
                inflight[c].append((op[1], op[2]))
            elif op[0] == "do":
                acts[op[1]] += 1
            elif op[0] == "need":
                for cond in op[1]:
                    if cond[0] == "mma" and cond[1] not in mdone:
                        return f"hazard at {op[2]} ({c}): product {cond[1]} not complete"
                    if cond[0] == "did" and acts[cond[1]] < cond[2]:
                        return f"hazard at {op[2]} ({c}): {cond[1]} done by {acts[cond[1]]} of {cond[2]}"
            cur[c] = next(self.progs[c], None)


def counts(ns):
    c = {("PFREE",): 2, ("WREADY",): 4, ("OFREE",): 4, ("MREADY",): 2, ("QREADY", 0): 2, ("QREADY", 1): 2,
         ("DLREADY",): 8}
    for s in range(ns):
        c[("EMPTY", s)] = 2
    return c


def state_roles(n, NG, g2, skip, NS=None, kda=False):
    """State warps 8..15; lane 0 of warp 8 issues Delta, O1, P_S and O2.
    Per-dim gate: no gate slots (the decay comes with the stage, copied out
    in the Delta epilogue)."""
    NS = NS or (2 if g2 else 3)
    def state(wi):
        issuer = wi == 0
        yield ("do", "put0")
        yield ("bar",)
        for ch in range(n):
            if issuer:
                yield ("wait", ("WREADY",), ch)
                yield ("wait", ("UFULL",), ch)
                yield ("need", [("did", f"wbw{ch}", 4), ("mma", f"U{ch}"), ("did", f"put{ch}", 8)], f"Delta {ch}")
                yield ("mma", f"D{ch}", [("WBFREE",), ("DLFULL",)])
                if ch >= 1 and skip != "OFREE":
                    yield ("wait", ("OFREE",), ch - 1)
                yield ("wait", ("QREADY", ch & 1), ch >> 1)
                yield ("need", [("did", f"qscale{ch}", 2), ("did", f"put{ch}", 8)] +
                       ([("did", f"oread{ch - 1}", 4)] if ch >= 1 else []), f"O1 {ch}")
                yield ("mma", f"O1_{ch}", [])
            if not kda:
                yield ("wait", ("GATE", ch % NG), ch // NG)
            yield ("wait", ("DLFULL",), ch)
            yield ("need", [("mma", f"D{ch}")] + ([("mma", f"O2_{ch - 1}")] if ch >= 1 else []), f"Delta epilogue {ch}")
            yield ("do", f"dlread{ch}")
            yield ("do", f"dbw{ch}")
            if kda and wi == 0:   # warp 8 keeps the chunk's decay past the stage's release
                yield ("need", [("did", f"load{ch}", 1)], f"decay copy {ch}")
                yield ("do", f"gcopy{ch}")
            yield ("arrive", ("DLREADY",))
            yield ("bar",)
            if issuer:
                yield ("need", [("did", f"dlread{ch}", 8), ("did", f"dbw{ch}", 8)], f"P_S {ch}")
                yield ("mma", f"PS{ch}", [("PSFULL",)])
                if skip != "MREADY":
                    yield ("wait", ("MREADY",), ch)
                yield ("need", [("did", f"maskw{ch}", 4 if g2 else 2), ("did", f"dbw{ch}", 8)], f"O2 {ch}")
                yield ("mma", f"O2_{ch}", [("OFULL",), ("MFREE",)])
                yield ("mma", f"E{ch}i", [("EMPTY", ch % NS)])
            yield ("wait", ("PSFULL",), ch)
            yield ("need", [("mma", f"PS{ch}"), ("mma", f"O1_{ch}")], f"state update {ch}")
            yield ("do", f"put{ch + 1}")
            yield ("bar",)
    return {f"state{i}": state(i) for i in range(8)}


def wepi_roles(n):
    """W/O epilogue warps 4..7: W of chunk t+1 first, then O of chunk t."""
    def wepi(wi):
        def w_epi(t):
            yield ("wait", ("WFULL",), t)
            yield ("need", [("mma", f"W{t}")], f"W epilogue {t}")
            yield ("do", f"wread{t}")
            if t >= 1:
                yield ("wait", ("WBFREE",), t - 1)
            yield ("need", [("mma", f"D{t - 1}")] if t >= 1 else [], f"W tile {t}")
            yield ("do", f"wbw{t}")
            yield ("arrive", ("WREADY",))
        yield from w_epi(0)
        for t in range(n):
            if t + 1 < n:
                yield from w_epi(t + 1)
            yield ("wait", ("OFULL",), t)
            yield ("need", [("mma", f"O1_{t}"), ("mma", f"O2_{t}")], f"O epilogue {t}")
            yield ("do", f"oread{t}")
            yield ("arrive", ("OFREE",))
    return {f"wepi{i}": wepi(i) for i in range(4)}


def producer_role(n, NS, stage_reads):
    NG = NS + 2

    def producer():
        yield ("arrive", ("GATE", 0))
        for t in range(n):
            if t >= NS:
                yield ("wait", ("EMPTY", t % NS), t // NS - 1)
                yield ("need", stage_reads(t - NS), f"load {t}")
            yield ("do", f"load{t}")
            yield ("arrive", ("FULL", t % NS))
            if t + 1 < n:
                yield ("arrive", ("GATE", (t + 1) % NG))
    return producer()


def single_head(n, skip=None):
    NS, NG = 3, 5

    def mma():
        for t in range(n):
            yield ("wait", ("FULL", t % NS), t // NS)
            if t >= 1:
                yield ("wait", ("WREADY",), t - 1)
                yield ("wait", ("WBFREE",), t - 1)
                if skip != "PFREE":
                    yield ("wait", ("PFREE",), t - 1)
            yield ("need", [("did", f"load{t}", 1)] + ([("did", f"pread{t - 1}", 2), ("did", f"wread{t - 1}", 4)]
                                                       if t >= 1 else []), f"QK, W {t}")
            yield ("mma", f"QK{t}", [("PFULL",)])
            yield ("mma", f"W{t}", [("WFULL",)])
            if t >= 1:
                yield ("wait", ("DLREADY",), t - 1)
            yield ("need", [("did", f"dlread{t - 1}", 8)] if t >= 1 else [], f"U {t}")
            yield ("mma", f"U{t}", [("UFULL",), ("EMPTY", t % NS)])

    def mask(wi):
        for ch in range(n):
            yield ("wait", ("GATE", ch % NG), ch // NG)
            yield ("wait", ("PFULL",), ch)
            yield ("need", [("mma", f"QK{ch}")], f"mask {ch}")
            yield ("do", f"qscale{ch}")
            yield ("arrive", ("QREADY", ch & 1))
            yield ("do", f"pread{ch}")
            yield ("arrive", ("PFREE",))
            if ch >= 1:
                yield ("wait", ("MFREE",), ch - 1)
            yield ("need", [("mma", f"O2_{ch - 1}")] if ch >= 1 else [], f"mask tile {ch}")
            yield ("do", f"maskw{ch}")
            yield ("arrive", ("MREADY",))

    def reads(u):
        return [("mma", x) for x in (f"QK{u}", f"W{u}", f"U{u}", f"O1_{u}", f"PS{u}")]

    progs = {"prod": producer_role(n, NS, reads), "mma": mma()}
    progs.update({f"mask{i}": mask(i) for i in range(2)})
    progs.update(wepi_roles(n))
    progs.update(state_roles(n, NG, False, skip))
    return progs, counts(NS)


def two_heads(n, skip=None):
    NS, NG = 2, 4

    def mma():
        for t in range(n):
            yield ("wait", ("FULL", t % NS), t // NS)
            if t >= 1:
                yield ("wait", ("WBFREE",), t - 1)
                if skip != "PFREE1":
                    yield ("wait", ("PFREE",), 2 * t - 1)
            yield ("need", [("did", f"load{t}", 1)] + ([("did", f"pread1_{t - 1}", 2)] if t >= 1 else []), f"W {t}")
            yield ("mma", f"W{t}", [("WFULL",)])
            if t >= 1:
                yield ("wait", ("DLREADY",), t - 1)
            yield ("need", [("did", f"dlread{t - 1}", 8)] if t >= 1 else [], f"U {t}")
            yield ("mma", f"U{t}", [("UFULL",)])
            if skip != "WREADY":
                yield ("wait", ("WREADY",), t)
            yield ("need", [("did", f"wread{t}", 4)], f"Q0 K^T {t}")
            yield ("mma", f"QK0_{t}", [("PFULL",)])
            if skip != "PFREE0":
                yield ("wait", ("PFREE",), 2 * t)
            yield ("need", [("did", f"pread0_{t}", 2)], f"Q1 K^T {t}")
            yield ("mma", f"QK1_{t}", [("PFULL",)])
            yield ("mma", f"E{t}", [("EMPTY", t % NS)])

    def mask(wi):
        for ch in range(n):
            yield ("wait", ("GATE", ch % NG), ch // NG)
            for hh in range(2):
                yield ("wait", ("PFULL",), 2 * ch + hh)
                yield ("need", [("mma", f"QK{hh}_{ch}")], f"mask {hh} {ch}")
                if hh == 1:
                    yield ("need", [("mma", f"QK0_{ch}"), ("mma", f"QK1_{ch}")], f"Q scaling {ch}")
                    yield ("do", f"qscale{ch}")
                    yield ("arrive", ("QREADY", ch & 1))
                yield ("do", f"pread{hh}_{ch}")
                yield ("arrive", ("PFREE",))
                if hh == 0 and ch >= 1:
                    yield ("wait", ("MFREE",), ch - 1)
                yield ("need", [("mma", f"O2_{ch - 1}")] if ch >= 1 else [], f"mask tile {hh} {ch}")
                yield ("do", f"maskw{ch}")
            yield ("arrive", ("MREADY",))

    def reads(u):
        return [("mma", x) for x in (f"W{u}", f"U{u}", f"QK0_{u}", f"QK1_{u}", f"O1_{u}", f"PS{u}")] + \
               [("did", f"qscale{u}", 2)]

    progs = {"prod": producer_role(n, NS, reads), "mma": mma()}
    progs.update({f"mask{i}": mask(i) for i in range(2)})
    progs.update(wepi_roles(n))
    progs.update(state_roles(n, NG, True, skip))
    return progs, counts(NS)


def preprocess(n, skip=None, role_s=True):
    """The pre-process chains (MODE_PRE, S role with U = T'V, M role with
    U = 0): lane 0 of warp 2 issues Delta and P_S and joins the state warps'
    named barrier; the MMA warp issues W (and U after the previous P_S)."""
    NS, NG = 3, 5

    def mma():
        for t in range(n):
            yield ("wait", ("FULL", t % NS), t // NS)
            if t >= 1:
                yield ("wait", ("WREADY",), t - 1)
                if skip != "WBFREE":   # W behind the chain's Delta (which then has read the W tile)
                    yield ("wait", ("WBFREE",), t - 1)
            yield ("need", [("did", f"load{t}", 1)] + ([("did", f"wread{t - 1}", 4)] if t >= 1 else []), f"W {t}")
            yield ("mma", f"W{t}", [("WFULL",)] + ([] if role_s else [("EMPTY", t % NS)]))
            if role_s:
                if t >= 1:
                    yield ("wait", ("DLREADY",), t - 1)
                    yield ("wait", ("PSFULL",), t - 1)   # scheduling: U behind the previous P_S
                yield ("need", [("did", f"dlread{t - 1}", 8)] if t >= 1 else [], f"U {t}")
                yield ("mma", f"U{t}", [("UFULL",), ("EMPTY", t % NS)])

    def wepi(wi):
        for t in range(n):
            yield ("wait", ("WFULL",), t)
            yield ("need", [("mma", f"W{t}")], f"W epilogue {t}")
            yield ("do", f"wread{t}")
            if t >= 1 and skip != "WBFREE":
                yield ("wait", ("WBFREE",), t - 1)
            yield ("need", [("mma", f"D{t - 1}")] if t >= 1 else [], f"W tile {t}")
            yield ("do", f"wbw{t}")
            yield ("arrive", ("WREADY",))

    def issuer():
        yield ("bar",)
        for ch in range(n):
            if skip != "WREADY":
                yield ("wait", ("WREADY",), ch)
            if role_s and skip != "UFULL":
                yield ("wait", ("UFULL",), ch)
            yield ("need", [("did", f"wbw{ch}", 4), ("did", f"put{ch}", 8)] + ([("mma", f"U{ch}")] if role_s else []),
                   f"Delta {ch}")
            yield ("mma", f"D{ch}", [("WBFREE",), ("DLFULL",)])
            yield ("bar",)
            yield ("need", [("did", f"dbw{ch}", 8), ("did", f"dlread{ch}", 8)] +
                   ([("did", f"psread{ch - 1}", 8)] if ch >= 1 else []), f"P_S {ch}")
            yield ("mma", f"PS{ch}", [("PSFULL",), ("EMPTY", ch % NS)])
            yield ("bar",)

    def state(wi):
        yield ("do", "put0")
        yield ("bar",)
        for ch in range(n):
            yield ("wait", ("GATE", ch % NG), ch // NG)
            yield ("wait", ("DLFULL",), ch)
            yield ("need", [("mma", f"D{ch}")] + ([("mma", f"PS{ch - 1}")] if ch >= 1 else []), f"Delta epilogue {ch}")
            yield ("do", f"dlread{ch}")
            yield ("do", f"dbw{ch}")
            if role_s:
                yield ("arrive", ("DLREADY",))
            yield ("bar",)
            yield ("wait", ("PSFULL",), ch)
            yield ("need", [("mma", f"PS{ch}"), ("mma", f"D{ch}")], f"state update {ch}")
            yield ("do", f"psread{ch}")
            yield ("do", f"put{ch + 1}")
            yield ("bar",)

    def reads(u):
        return [("mma", x) for x in ([f"W{u}", f"PS{u}"] + ([f"U{u}"] if role_s else []))]

    progs = {"prod": producer_role(n, NS, reads), "mma": mma(), "state_issuer": issuer()}
    progs.update({f"wepi{i}": wepi(i) for i in range(4)})
    progs.update({f"state{i}": state(i) for i in range(8)})
    return progs, counts(NS)


def preprocess_m(n, skip=None):
    return preprocess(n, skip, role_s=False)


def single_head_kda(n, skip=None):
    """The per-dim gate's forward (MODE_FWD_KDA): the unit's pre-gated Qg and
    P arrive with the stage (two stages), the mask warps only release them
    one chunk ahead, no Q K^T product and no gate slots."""
    NS = 2

    def mma():
        for t in range(n):
            yield ("wait", ("FULL", t % NS), t // NS)
            if t >= 1:
                yield ("wait", ("WREADY",), t - 1)
                yield ("wait", ("WBFREE",), t - 1)
            yield ("need", [("did", f"load{t}", 1)] + ([("did", f"wread{t - 1}", 4)] if t >= 1 else []), f"W {t}")
            yield ("mma", f"W{t}", [("WFULL",)])
            if t >= 1 and skip != "DLREADY":
                yield ("wait", ("DLREADY",), t - 1)
            yield ("need", [("did", f"dlread{t - 1}", 8)] if t >= 1 else [], f"U {t}")
            yield ("mma", f"U{t}", [("UFULL",), ("EMPTY", t % NS)])

    def mask(wi):
        for ch in range(n):
            if ch >= 1 and skip != "MFREE":
                yield ("wait", ("MFREE",), ch - 1)
            yield ("wait", ("FULL", ch % NS), ch // NS)
            yield ("do", f"qscale{ch}")     # releases the stage's Qg
            yield ("arrive", ("QREADY", ch & 1))
            yield ("do", f"maskw{ch}")      # and its P
            yield ("arrive", ("MREADY",))

    def producer():
        for t in range(n):
            if t >= NS:
                yield ("wait", ("EMPTY", t % NS), t // NS - 1)
                u = t - NS
                yield ("need", [("mma", x) for x in (f"W{u}", f"U{u}", f"O1_{u}", f"PS{u}", f"O2_{u}")] +
                       [("did", f"gcopy{u}", 1)], f"load {t}")
            yield ("do", f"load{t}")
            yield ("arrive", ("FULL", t % NS))

    progs = {"prod": producer(), "mma": mma()}
    progs.update({f"mask{i}": mask(i) for i in range(2)})
    progs.update(wepi_roles(n))
    progs.update(state_roles(n, 0, False, skip, NS=NS, kda=True))
    return progs, counts(NS)


def backward(n, skip=None):
    """The state-gradient chain (MODE_BWD, scalar gate), chunks in reverse:
    per chunk the issuing lane of warp 8 issues X1 = dO^T mask (into the
    Delta columns) and X2 = dS'^T K^T (into the output columns), the state
    warps form dDelta from both and write -dDelta^T, then X3 + X4 =
    dO^T (gamma ⊙ Q) - dDelta^T W (into the P_S columns) updates dS.  The
    MMA warp issues Q K^T and W as in the forward (no U)."""
    NS, NG = 3, 5

    def mma():
        for t in range(n):
            yield ("wait", ("FULL", t % NS), t // NS)
            if t >= 1:
                yield ("wait", ("WREADY",), t - 1)
                if skip != "WBFREE":
                    yield ("wait", ("WBFREE",), t - 1)
                yield ("wait", ("PFREE",), t - 1)
            yield ("need", [("did", f"load{t}", 1)] + ([("did", f"pread{t - 1}", 2), ("did", f"wread{t - 1}", 4)]
                                                       if t >= 1 else []), f"QK, W {t}")
            yield ("mma", f"QK{t}", [("PFULL",)])
            yield ("mma", f"W{t}", [("WFULL",), ("EMPTY", t % NS)])

    def mask(wi):
        for ch in range(n):
            yield ("wait", ("GATE", ch % NG), ch // NG)
            yield ("wait", ("PFULL",), ch)
            yield ("need", [("mma", f"QK{ch}")], f"mask {ch}")
            yield ("do", f"qscale{ch}")
            yield ("arrive", ("QREADY", ch & 1))
            yield ("do", f"pread{ch}")
            yield ("arrive", ("PFREE",))
            if ch >= 1:
                yield ("wait", ("MFREE",), ch - 1)
            yield ("need", [("mma", f"X1_{ch - 1}")] if ch >= 1 else [], f"mask tile {ch}")
            yield ("do", f"maskw{ch}")
            yield ("arrive", ("MREADY",))

    def wepi(wi):
        for t in range(n):
            yield ("wait", ("WFULL",), t)
            yield ("need", [("mma", f"W{t}")], f"W epilogue {t}")
            yield ("do", f"wread{t}")
            if t >= 1 and skip != "WBFREE":
                yield ("wait", ("WBFREE",), t - 1)
            yield ("need", [("mma", f"X34_{t - 1}")] if t >= 1 else [], f"W tile {t}")
            yield ("do", f"wbw{t}")
            yield ("arrive", ("WREADY",))

    def state(wi):
        issuer = wi == 0
        yield ("do", "put0")
        yield ("bar",)
        for t in range(n):
            if issuer:
                if skip != "MREADY":
                    yield ("wait", ("MREADY",), t)
                yield ("need", [("did", f"maskw{t}", 2), ("did", f"put{t}", 8)] +
                       ([("did", f"dlread{t - 1}", 8)] if t >= 1 else []), f"X1, X2 {t}")
                yield ("mma", f"X1_{t}", [("MFREE",)])
                yield ("mma", f"X2_{t}", [("DLFULL",)])
            yield ("wait", ("GATE", t % NG), t // NG)
            yield ("wait", ("DLFULL",), t)
            yield ("need", [("mma", f"X1_{t}"), ("mma", f"X2_{t}")] +
                   ([("mma", f"X34_{t - 1}")] if t >= 1 else []), f"dDelta {t}")
            yield ("do", f"dlread{t}")
            yield ("do", f"dbw{t}")
            yield ("bar",)
            if issuer:
                yield ("wait", ("QREADY", t & 1), t >> 1)
                if skip != "WREADY":
                    yield ("wait", ("WREADY",), t)
                yield ("need", [("did", f"qscale{t}", 2), ("did", f"wbw{t}", 4), ("did", f"dbw{t}", 8)] +
                       ([("did", f"psread{t - 1}", 8)] if t >= 1 else []), f"X3, X4 {t}")
                yield ("mma", f"X34_{t}", [("PSFULL",), ("WBFREE",)])
                yield ("mma", f"E{t}i", [("EMPTY", t % NS)])
            yield ("wait", ("PSFULL",), t)
            yield ("need", [("mma", f"X34_{t}"), ("mma", f"X2_{t}")], f"dS update {t}")
            yield ("do", f"psread{t}")
            yield ("do", f"put{t + 1}")
            yield ("bar",)

    def reads(u):
        return [("mma", x) for x in (f"QK{u}", f"W{u}", f"X1_{u}", f"X2_{u}", f"X34_{u}")] + [("did", f"qscale{u}", 2)]

    progs = {"prod": producer_role(n, NS, reads), "mma": mma()}
    progs.update({f"mask{i}": mask(i) for i in range(2)})
    progs.update({f"wepi{i}": wepi(i) for i in range(4)})
    progs.update({f"state{i}": state(i) for i in range(8)})
    return progs, counts(NS)


MODELS = {"single_head": single_head, "two_heads": two_heads, "single_head_kda": single_head_kda,
          "pre_s": preprocess, "pre_m": preprocess_m, "backward": backward}
MUTATIONS = {"single_head": ["PFREE", "OFREE", "MREADY"],
             "two_heads": ["PFREE0", "PFREE1", "WREADY", "OFREE", "MREADY"],
             "single_head_kda": ["OFREE", "DLREADY", "MFREE"],
             "pre_s": ["WBFREE", "UFULL", "WREADY"],
             "pre_m": ["WBFREE", "WREADY"],
             "backward": ["WBFREE", "MREADY", "WREADY"]}


def failures(model, skip, seeds):
    out = []
    for n in (1, 2, 3, 4, 7):
        for seed in range(seeds):
            progs, cnt = MODELS[model](n, skip)
            e = Protocol(progs, cnt, seed).run()
            if e:
                out.append((n, seed, e))
    return out


@pytest.mark.parametrize("model", list(MODELS))
def test_protocol_has_no_deadlock_or_hazard(model):
    bad = failures(model, None, 120)
    assert not bad, bad[:3]


@pytest.mark.parametrize("model,skip", [(m, s) for m in MODELS for s in MUTATIONS[m]])
def test_checker_catches_a_missing_wait(model, skip):
    assert failures(model, skip, 120), f"removing the {skip} wait went unnoticed"
