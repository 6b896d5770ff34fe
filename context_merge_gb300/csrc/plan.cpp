// Host planner: cuts rows (or a packed batch) into R contiguous segments and
// lists every local fragment with its role in the segmented scheme.
//
// Follows the article "flash-linear-attention 上下文并行CP ..." ([FLA-CP]):
//   §3.2  contiguous layout: segment r holds tokens [r*T/R, (r+1)*T/R);
//         zigzag layout: 2R equal parts, rank r holding parts r and 2R-1-r
//   §3.3  total tokens must be >= R and divisible by R (ValueError there,
//         CPDR_ERR_INVALID here); sequences intersecting a segment are found
//         by a sorted search over the global cu_seqlens and truncated to it
//   §5.2  the forward merge feeds a segment's FIRST local sequence; the
//         pre-process covers its LAST local sequence when that one continues
#include <algorithm>
#include <cstdio>
#include <numeric>

#include "cpdr_internal.hpp"

namespace cpdr {

static cpdr_status fail(std::string &err, cpdr_status s, const char *msg) {
    err = msg;
    return s;
}

cpdr_status build_plan(const cpdr_desc &d, Plan &p, std::string &err) {
    if (d.B < 1 || d.H < 1 || d.dk < 1 || d.dv < 1 || d.R < 1 || d.T < 1)
        return fail(err, CPDR_ERR_INVALID, "B, H, dk, dv, R and T must be positive");
    if (d.gate_kind != CPDR_GATE_SCALAR && d.gate_kind != CPDR_GATE_PER_DIM)
        return fail(err, CPDR_ERR_INVALID, "gate_kind must be CPDR_GATE_SCALAR or CPDR_GATE_PER_DIM");
    if (d.in_dtype != CPDR_DTYPE_F32 && d.in_dtype != CPDR_DTYPE_BF16)
        return fail(err, CPDR_ERR_INVALID, "in_dtype must be CPDR_DTYPE_F32 or CPDR_DTYPE_BF16");
    if (d.dk != d.dv || (d.dk != 64 && d.dk != 128))
        return fail(err, CPDR_ERR_UNSUPPORTED, "only dk == dv in {64, 128} is implemented");
    if (d.conv_width < 0 || d.conv_width > kMaxConvWidth)
        return fail(err, CPDR_ERR_UNSUPPORTED, "conv_width must be 0 (no conv path) or 1..8");
    if (d.Hq != 0 && (d.Hq < d.H || d.Hq % d.H != 0))
        return fail(err, CPDR_ERR_INVALID, "Hq must be 0, H, or a multiple of H (grouped query heads)");
    // zigzag placement ([FLA-CP] §3.2): 2R pieces, rank r holding pieces r and
    // 2R-1-r; on one GPU every piece is a segment of its own, in sequence order
    const bool zigzag = (d.flags & CPDR_FLAG_LAYOUT_ZIGZAG) != 0;
    const int64_t pieces = zigzag ? 2 * (int64_t)d.R : d.R;
    if (pieces > INT32_MAX / 2) return fail(err, CPDR_ERR_INVALID, "R too large");
    if (d.T % pieces != 0 || d.T < pieces)
        return fail(err, CPDR_ERR_INVALID,
                    zigzag ? "tokens per row (or packed total) must be >= 2R and divisible by 2R (zigzag layout)"
                           : "tokens per row (or packed total) must be >= R and divisible by R");
    if (d.T > (int64_t)INT32_MAX * kChunk)
        return fail(err, CPDR_ERR_INVALID, "too many tokens");

    p = Plan();
    p.B = d.B; p.H = d.H; p.dk = d.dk; p.dv = d.dv; p.R = (int32_t)pieces; p.T = d.T;
    p.gate_kind = d.gate_kind; p.in_dtype = d.in_dtype; p.flags = d.flags; p.scale = d.scale;
    p.L = d.T / pieces;
    p.Hq = d.Hq ? d.Hq : d.H;
    p.G = p.Hq / p.H;
    p.vfirst = (d.flags & CPDR_FLAG_STATE_V_FIRST) != 0;
    p.conv_width = d.conv_width;
    if (p.L > INT32_MAX) return fail(err, CPDR_ERR_INVALID, "segment length exceeds 2^31-1");

    if (d.cu_seqlens_host) {
        if (d.B != 1) return fail(err, CPDR_ERR_INVALID, "packed batches (cu_seqlens) need B == 1");
        if (d.num_seqs < 1) return fail(err, CPDR_ERR_INVALID, "num_seqs must be >= 1");
        p.packed = true;
        p.N = d.num_seqs;
        p.cu.assign(d.cu_seqlens_host, d.cu_seqlens_host + d.num_seqs + 1);
        if (p.cu[0] != 0 || p.cu[p.N] != d.T)
            return fail(err, CPDR_ERR_INVALID, "cu_seqlens must start at 0 and end at T");
        for (int n = 0; n < p.N; n++)
            if (p.cu[n + 1] < p.cu[n]) return fail(err, CPDR_ERR_INVALID, "cu_seqlens must be non-decreasing");
    } else {
        if (d.num_seqs != 0 && d.num_seqs != d.B)
            return fail(err, CPDR_ERR_INVALID, "num_seqs must equal B (or 0) without cu_seqlens");
        p.N = d.B;
        p.cu.resize(p.N + 1);
        for (int n = 0; n <= p.N; n++) p.cu[n] = (int64_t)n * d.T;
    }

    // Fragments: for row b and segment r, intersect [base + r L, base + (r+1) L)
    // with the sequences.  Fixed-length rows are one sequence each.  Segments
    // and sequences live in sequence coordinates; tok0 is where a fragment's
    // tokens are in memory: the same place in the contiguous layout, and in
    // the zigzag layout part r sits at slot 2r (r < R) or 2(2R-1-r)+1 of its
    // row, rank by rank, each rank's [front; back]
    const int64_t L = p.L;
    auto mem_slot = [&](int r) -> int64_t {
        if (!zigzag) return r;
        return r < d.R ? 2 * (int64_t)r : 2 * (int64_t)(2 * d.R - 1 - r) + 1;
    };
    std::vector<int32_t> first_frag_of_seg(p.nseg(), -1), last_frag_of_seg(p.nseg(), -1);
    std::vector<int32_t> frag_halo;   // conv halo row of each fragment (or kHaloZero)
    const int halo_w = d.conv_width > 0 ? d.conv_width - 1 : 0;
    if (d.conv_width > 0) p.conv_pre_tokens.assign(p.nseg(), 0);
    // memory position of sequence position x of row b (base = the row's start)
    auto mem_of = [&](int64_t base, int64_t x) {
        const int64_t off = x - base;
        return base + mem_slot((int)(off / L)) * L + off % L;
    };
    for (int b = 0; b < p.B; b++) {
        const int64_t base = p.packed ? 0 : (int64_t)b * p.T;
        for (int r = 0; r < p.R; r++) {
            const int64_t s0 = base + (int64_t)r * L, s1 = s0 + L;
            const int32_t seg = r * p.B + b;
            // first sequence whose end lies beyond s0 (upper_bound on cu[1..N])
            int n = (int)(std::upper_bound(p.cu.begin() + 1, p.cu.end(), s0) - (p.cu.begin() + 1));
            for (; n < p.N && p.cu[n] < s1; n++) {
                const int64_t a = std::max(p.cu[n], s0), e = std::min(p.cu[n + 1], s1);
                if (e <= a) continue;  // zero-length sequence
                cpdr_fragment f;
                f.tok0 = base + mem_slot(r) * L + (a - s0);
                f.len = (int32_t)(e - a);
                f.seg = seg;
                f.seq = n;
                f.flags = 0;
                if (p.cu[n] < s0) f.flags |= CPDR_FRAG_CONT_PREV;
                if (p.cu[n + 1] > s1) f.flags |= CPDR_FRAG_CONT_NEXT;
                else f.flags |= CPDR_FRAG_ENDS_SEQ;
                // causal conv1d ([FLA-CP] §2.4, §3.3): a segment's first
                // fragment that continues a sequence reads the conv_width - 1
                // inputs before it, in sequence order (wherever they are in
                // memory), down to the sequence start: pre_num_conv_tokens
                int32_t halo = kHaloZero;
                if (d.conv_width > 0 && (f.flags & CPDR_FRAG_CONT_PREV)) {
                    halo = (int32_t)(p.conv_halo.size() / std::max(halo_w, 1));
                    const int64_t avail = a - p.cu[n];
                    p.conv_pre_tokens[seg] = (int32_t)std::min<int64_t>(halo_w, avail);
                    for (int j = halo_w; j >= 1; j--)   // oldest first
                        p.conv_halo.push_back(j <= avail ? mem_of(base, a - j) : -1);
                    if (halo_w == 0) halo = kHaloZero;
                }
                frag_halo.push_back(halo);
                if (first_frag_of_seg[seg] < 0) first_frag_of_seg[seg] = (int32_t)p.frags.size();
                last_frag_of_seg[seg] = (int32_t)p.frags.size();
                p.frags.push_back(f);
            }
        }
    }
    for (int n = 0; n < p.N; n++)
        if (p.cu[n + 1] == p.cu[n]) p.empty_seqs.push_back(n);

    for (int32_t s = 0; s < p.nseg(); s++) {
        const int32_t lf = last_frag_of_seg[s], ff = first_frag_of_seg[s];
        if (lf >= 0 && (p.frags[lf].flags & CPDR_FRAG_CONT_NEXT)) p.pre_items.push_back(lf);
        else p.zero_pre.push_back(s);
        if (!(ff >= 0 && (p.frags[ff].flags & CPDR_FRAG_CONT_PREV))) p.zero_init.push_back(s);
    }
    // Merge chains: one per sequence crossing at least one cut.
    for (int n = 0; n < p.N; n++) {
        if (p.cu[n + 1] == p.cu[n]) continue;
        const int b = p.packed ? 0 : n;
        const int64_t base = p.packed ? 0 : (int64_t)b * p.T;
        const int r0 = (int)((p.cu[n] - base) / L), r1 = (int)((p.cu[n + 1] - 1 - base) / L);
        if (r1 > r0) p.chains.push_back(MergeChain{b, r0, r1, 0});
    }
    auto chunks = [](int32_t len) { return (len + kChunk - 1) / kChunk; };
    for (int32_t i : p.pre_items) p.max_pre_chunks = std::max(p.max_pre_chunks, chunks(p.frags[i].len));
    p.fwd_order.resize(p.frags.size());
    std::iota(p.fwd_order.begin(), p.fwd_order.end(), 0);
    std::stable_sort(p.fwd_order.begin(), p.fwd_order.end(),
                     [&](int32_t a, int32_t b) { return p.frags[a].len > p.frags[b].len; });
    for (auto &f : p.frags) p.max_fwd_chunks = std::max(p.max_fwd_chunks, chunks(f.len));
    // host-buffer pipeline: fragments in memory order (they tile the token
    // axis), cut at fragment boundaries into kHostParts groups of about
    // equal tokens; longest first inside a group
    {
        std::vector<int32_t> mem(p.frags.size());
        std::iota(mem.begin(), mem.end(), 0);
        std::stable_sort(mem.begin(), mem.end(),
                         [&](int32_t a, int32_t b) { return p.frags[a].tok0 < p.frags[b].tok0; });
        const int64_t total = (int64_t)p.B * p.T;
        std::vector<std::vector<int32_t>> groups(kHostParts);
        int g = 0;
        int64_t acc = 0;
        for (int32_t fi : mem) {
            while (g + 1 < kHostParts && acc >= (int64_t)(g + 1) * total / kHostParts) g++;
            groups[g].push_back(fi);
            acc += p.frags[fi].len;
        }
        int64_t cursor = 0;
        for (int gi = 0; gi < kHostParts; gi++) {
            std::stable_sort(groups[gi].begin(), groups[gi].end(),
                             [&](int32_t a, int32_t b) { return p.frags[a].len > p.frags[b].len; });
            p.host_part_off[gi] = (int32_t)p.host_items.size();
            p.host_part_tok[gi] = cursor;
            for (int32_t fi : groups[gi]) {
                p.host_items.push_back(fi);
                cursor += p.frags[fi].len;
            }
        }
        p.host_part_off[kHostParts] = (int32_t)p.host_items.size();
        p.host_part_tok[kHostParts] = cursor;
        if (cursor != total) return fail(err, CPDR_ERR_INVALID, "internal: fragments do not tile the token axis");
    }
    for (size_t i = 0; i < p.frags.size(); i++)
        if (p.frags[i].flags & CPDR_FRAG_CONT_PREV) p.bwd_pre_items.push_back((int32_t)i);
    // longest pre items first as well
    std::stable_sort(p.pre_items.begin(), p.pre_items.end(),
                     [&](int32_t a, int32_t b) { return p.frags[a].len > p.frags[b].len; });
    // every chunk of every fragment, fragment by fragment (the WY tiles'
    // order): fragment f's chunk c is global chunk frag_chunk0[f] + c
    p.frag_chunk0.resize(p.frags.size() + 1);
    int32_t acc = 0;
    for (size_t i = 0; i < p.frags.size(); i++) {
        const cpdr_fragment &f = p.frags[i];
        p.frag_chunk0[i] = acc;
        for (int32_t c = 0; c < chunks(f.len); c++)
            p.wy_chunks.push_back(WyChunk{f.tok0 + (int64_t)c * kChunk, std::min(kChunk, f.len - c * kChunk), 0});
        acc += chunks(f.len);
    }
    p.frag_chunk0.back() = acc;
    if (d.conv_width > 0) {
        for (size_t i = 0; i < p.frags.size(); i++) {
            const cpdr_fragment &f = p.frags[i];
            for (int32_t c = 0; c < f.len; c += kConvTile)
                p.conv_tiles.push_back(ConvTile{f.tok0 + c, std::min(kConvTile, f.len - c),
                                                c > 0 ? kHaloMemory : frag_halo[i]});
        }
    }
    return CPDR_OK;
}

}  // namespace cpdr
