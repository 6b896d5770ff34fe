"""Host planner (segment/fragment tables) against the article's cut rules:
golden fragment tables for the test-matrix cut patterns and the debug
example (tests/golden/partitions.json, each with its citation), plus
structural properties on other patterns.  CPU only."""
import json
import os

import pytest

from context_merge_gb300 import cpdr

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "partitions.json")))


def ctx_for(lengths, R, H=1, d=64):
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    return cpdr.Context(B=1, T=cu[-1], H=H, d=d, R=R, gate="gdn", dtype="bf16", cu_seqlens=cu, host_only=True)


@pytest.mark.parametrize("case", GOLD["cases"], ids=[c["name"] for c in GOLD["cases"]])
def test_golden_fragments(cpdr_lib, case):
    frags = ctx_for(case["lengths"], case["R"]).fragments()
    assert [list(f) for f in frags] == case["fragments"]
    if "chunk_starts" in case:
        starts = [list(range(f[0], f[0] + f[1], 64)) for f in frags]
        assert starts == case["chunk_starts"]


@pytest.mark.parametrize("case", GOLD["invalid"], ids=[c["cite"] for c in GOLD["invalid"]])
def test_golden_invalid(cpdr_lib, case):
    with pytest.raises(cpdr.CpdrError) as ei:
        ctx_for(case["lengths"], case["R"])
    assert ei.value.status == cpdr.ERR_INVALID


def check_structure(frags, cu, R):
    T = cu[-1]
    L = T // R
    # fragments tile the token axis in order, never cross a segment or sequence boundary
    pos = 0
    for tok0, ln, seg, seq, fl in frags:
        assert tok0 == pos and ln >= 1
        pos += ln
        assert tok0 // L == seg and (tok0 + ln - 1) // L == seg
        assert cu[seq] <= tok0 and tok0 + ln <= cu[seq + 1]
        assert bool(fl & cpdr.FRAG_CONT_PREV) == (cu[seq] < tok0)
        assert bool(fl & cpdr.FRAG_ENDS_SEQ) == (tok0 + ln == cu[seq + 1])
        assert bool(fl & cpdr.FRAG_CONT_NEXT) == (tok0 + ln < cu[seq + 1])
    assert pos == T
    # only a segment's first fragment may continue, only its last may cross
    by_seg = {}
    for f in frags:
        by_seg.setdefault(f[2], []).append(f)
    for seg, fs in by_seg.items():
        for f in fs[1:]:
            assert not f[4] & cpdr.FRAG_CONT_PREV
        for f in fs[:-1]:
            assert not f[4] & cpdr.FRAG_CONT_NEXT


@pytest.mark.parametrize("lengths,R", [
    ([5, 7, 6, 9, 4, 11, 6, 16], 2),      # many short sequences
    ([64] * 8, 4),                         # cuts exactly on sequence starts
    ([100, 0, 28], 2),                     # an empty sequence
    ([1] * 64, 64),                        # one token per segment
    ([4097, 3, 4092], 4),
])
def test_structure(cpdr_lib, lengths, R):
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    check_structure(ctx_for(lengths, R).fragments(), cu, R)


def test_fixed_rows(cpdr_lib):
    ctx = cpdr.Context(B=3, T=256, H=1, d=64, R=4, gate="gdn", dtype="fp32", host_only=True)
    frags = ctx.fragments()
    assert len(frags) == 12
    for r in range(4):
        for b in range(3):
            f = frags[r * 3 + b] if False else [x for x in frags if x[2] == r * 3 + b][0]
            assert f[0] == b * 256 + r * 64 and f[1] == 64 and f[3] == b
            want = (cpdr.FRAG_CONT_PREV if r > 0 else 0) | (cpdr.FRAG_CONT_NEXT if r < 3 else cpdr.FRAG_ENDS_SEQ)
            assert f[4] == want


# ---- zigzag layout ([FLA-CP] §3.2) and grouped query heads (§5.1) ---------
def test_zigzag_worked_example(cpdr_lib):
    """One 8-token sequence, R = 2 ranks: parts [0,2) [2,4) [4,6) [6,8) sit in
    memory as rank 0 = [part 0; part 3], rank 1 = [part 1; part 2]."""
    ctx = cpdr.Context(B=1, T=8, H=1, d=64, R=2, gate="gdn", dtype="bf16", host_only=True, layout="zigzag")
    P, N, E = cpdr.FRAG_CONT_PREV, cpdr.FRAG_CONT_NEXT, cpdr.FRAG_ENDS_SEQ
    assert ctx.fragments() == [(0, 2, 0, 0, N), (4, 2, 1, 0, P | N), (6, 2, 2, 0, P | N), (2, 2, 3, 0, P | E)]
    assert ctx.pieces == 4
    sext, m, sinit, fin = ctx.buffer_sizes()
    assert sext == 4 * 1 * 1 * 64 * 64 * 4 and fin == 64 * 64 * 4


@pytest.mark.parametrize("lengths,R", [
    ([3000, 4000, 3240], 2),
    ([7000, 3240], 4),
    ([5, 7, 6, 9, 4, 11, 6, 16], 2),
    ([100, 0, 28], 2),
    ([4097, 3, 4092], 4),
    ([65536], 8),
])
def test_zigzag_is_the_contiguous_plan_of_2r_parts_moved(cpdr_lib, lengths, R):
    """Mapped back to sequence positions, the zigzag plan is the contiguous
    plan of 2R segments, and every fragment is contiguous in memory."""
    from oracle import layout
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    zz = cpdr.Context(B=1, T=cu[-1], H=1, d=64, R=R, gate="gdn", dtype="bf16", cu_seqlens=cu, host_only=True,
                      layout="zigzag").fragments()
    pos = layout.zigzag_positions(cu[-1], R)
    for tok0, ln, *_ in zz:
        assert (pos[tok0:tok0 + ln] == pos[tok0] + list(range(ln))).all()
    seq_order = [(int(pos[f[0]]),) + tuple(f[1:]) for f in zz]
    assert seq_order == ctx_for(lengths, 2 * R).fragments()
    check_structure(seq_order, cu, 2 * R)


def test_zigzag_fixed_rows(cpdr_lib):
    from oracle import layout
    B, T, R = 3, 256, 4
    zz = cpdr.Context(B=B, T=T, H=1, d=64, R=R, gate="gdn", dtype="fp32", host_only=True,
                      layout="zigzag").fragments()
    pos = layout.zigzag_positions(T, R)
    assert len(zz) == B * 2 * R
    for tok0, ln, seg, seq, fl in zz:
        b = tok0 // T
        r = seg // B
        assert seq == b and seg == r * B + b and ln == T // (2 * R)
        assert pos[tok0 - b * T] == r * ln


@pytest.mark.parametrize("T,R,ok", [(12, 4, False), (16, 4, True), (6, 4, False), (8, 4, True)])
def test_zigzag_cut_rule(cpdr_lib, T, R, ok):
    """[FLA-CP] §3.3: zigzag needs tokens >= 2R and divisible by 2R."""
    mk = lambda: cpdr.Context(B=1, T=T, H=1, d=64, R=R, gate="gdn", dtype="bf16", host_only=True, layout="zigzag")
    if ok:
        mk()
    else:
        with pytest.raises(cpdr.CpdrError) as ei:
            mk()
        assert ei.value.status == cpdr.ERR_INVALID


@pytest.mark.parametrize("H,Hq,ok", [(2, 4, True), (2, 2, True), (4, 12, True), (2, 3, False), (4, 2, False)])
def test_grouped_query_heads_validation(cpdr_lib, H, Hq, ok):
    mk = lambda: cpdr.Context(B=1, T=256, H=H, d=64, R=2, gate="gdn", dtype="bf16", host_only=True, Hq=Hq)
    if ok:
        sext, m, sinit, fin = mk().buffer_sizes()
        assert sext == 2 * H * 64 * 64 * 4 and fin == H * 64 * 64 * 4   # states keep H heads
    else:
        with pytest.raises(cpdr.CpdrError) as ei:
            mk()
        assert ei.value.status == cpdr.ERR_INVALID


# ---- causal conv1d halo ([FLA-CP] §2.4, §3.3 pre_num_conv_tokens) ----------
@pytest.mark.parametrize("lengths,R,W,zigzag", [
    ([3000, 4000, 3240], 2, 4, False),
    ([5118, 5122], 2, 4, False),
    ([7000, 3240], 4, 4, False),
    ([5, 7, 6, 9, 4, 11, 6, 16], 8, 8, False),
    ([1] * 64, 32, 4, False),
    ([100, 0, 28], 2, 3, True),
    ([3000, 4000, 3240], 4, 4, True),
    ([8], 2, 4, True),
    ([3, 5], 2, 3, True),
])
def test_pre_num_conv_tokens(cpdr_lib, lengths, R, W, zigzag):
    from oracle import conv
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    ctx = cpdr.Context(B=1, T=cu[-1], H=1, d=64, R=R, gate="gdn", dtype="bf16", cu_seqlens=cu, host_only=True,
                       layout="zigzag" if zigzag else "contiguous", conv_width=W)
    assert ctx.conv_pre_tokens() == conv.pre_num_conv_tokens(cu, cu[-1], R, W, zigzag=zigzag)


def test_conv_width_validation(cpdr_lib):
    mk = lambda W: cpdr.Context(B=1, T=256, H=1, d=64, R=2, gate="gdn", dtype="bf16", host_only=True,
                                conv_width=W)
    for W in (0, 1, 4, 8):
        mk(W)
    for W, st in ((9, cpdr.ERR_UNSUPPORTED), (-1, cpdr.ERR_UNSUPPORTED)):
        with pytest.raises(cpdr.CpdrError) as ei:
            mk(W)
        assert ei.value.status == st
    with pytest.raises(cpdr.CpdrError):
        mk(0).conv_pre_tokens()


# ---- seeded random length mixes: structure and the plan's counters -------
def _random_case(rng):
    R = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    L = int(rng.integers(1, 40))
    T = R * L
    n = int(rng.integers(1, 12))
    cuts = sorted(int(x) for x in rng.integers(0, T + 1, size=n - 1))
    bounds = [0] + cuts + [T]
    lengths = [bounds[i + 1] - bounds[i] for i in range(n)]
    return lengths, R


@pytest.mark.parametrize("seed", range(60))
def test_random_mixes_structure_and_counters(cpdr_lib, seed):
    rng = __import__("numpy").random.default_rng(5000 + seed)
    lengths, R = _random_case(rng)
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    T = cu[-1]
    L = T // R
    ctx = ctx_for(lengths, R)
    frags = ctx.fragments()
    check_structure(frags, cu, R)
    c = ctx.counts()
    assert c["fragments"] == len(frags)
    # the pre-process runs each segment's fragment that continues past it
    assert c["pre_items"] == sum(1 for f in frags if f[4] & cpdr.FRAG_CONT_NEXT)
    # one merge chain per sequence that spans at least two segments
    spans = [(cu[i] // L, (cu[i + 1] - 1) // L) for i in range(len(lengths)) if lengths[i] > 0]
    assert c["chains"] == sum(1 for a, b in spans if b > a)
    assert c["empty_seqs"] == sum(1 for x in lengths if x == 0)
    # S_ext/M are zeroed where no fragment continues; S_init where none is continued
    cont_next = {f[2] for f in frags if f[4] & cpdr.FRAG_CONT_NEXT}
    cont_prev = {f[2] for f in frags if f[4] & cpdr.FRAG_CONT_PREV}
    assert c["zero_pre"] == R - len(cont_next)
    assert c["zero_init"] == R - len(cont_prev)
