// Tensor-core (tcgen05 / TMEM / TMA) chain kernels for the bf16, d = 128
// path of the segmented delta-rule forward, scalar gate (GDN).
//
// One CTA runs one chain: a (fragment, head) pair, 64-token chunks in order.
// The per-chunk inverse T = (I + A)^-1 comes precomputed from the WY build
// (tc_wy.cu) as bf16 tiles T' = T diag(beta) and T'' = T diag(beta gamma)
// (hi, and lo for the split M chain).  Per chunk, following the chunk form of
// the article "flash-linear-attention 上下文并行CP ..." ([FLA-CP] §2.2) in
// transposed storage (state rows = value dims, so every product has M = 128
// on the tensor core):
//   W^T    = K^T T''^T,  U^T = V^T T'^T                      (MMA)
//   Delta^T= U^T - S^T W^T                                   (MMA, accumulate)
//   O^T    = S^T (gamma ⊙ Q)^T + Delta^T mask^T,  gamma_i = 2^(G_i),
//            mask_ij = (Q K^T)_ij 2^(G_i - G_j), j <= i      (forward)
//   S^T   <- gamma^C S^T + (Delta diag(Gamma))^T K,  Gamma_j = 2^(G_C - G_j)
// The pre-process runs the same chain without outputs (role S) and, in a
// second launch, the transfer-matrix chain
//   M <- M_[t] M,  M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W   ([FLA-CP] §2.2)
// (role M: U = 0, M_0 = I).  The M chain keeps fp32 accuracy, as the article
// requires: its accumulator lives in fp32 registers and every tensor-core
// operand derived from a rounded quantity (T'', W, M, Delta) is a bf16 hi/lo
// pair, so each product is hi*hi + lo*hi + hi*lo.
//
// Warp roles (16 warps): 0 TMA producer and in-chunk gates; 1 MMA issuer
// (+ TMEM owner); 2-3 causal mask (forward only); 4-7 W and O epilogues;
// 8-15 state warps (Delta epilogue and S update; the fp32 state lives in
// their registers, 64 values per thread).  The critical path per chunk is
//   Delta MMA -> Delta epilogue -> P_S MMA -> S update -> Delta MMA,
// and the next chunk's W, U (and Q K^T) products are issued into the gaps.
// Roles and shared-memory layouts are compile-time and every role function
// is inlined, so per-CTA state stays in registers.  Every mbarrier wait is
// bounded: on expiry the kernel records a status code, raises an abort flag
// that makes every other wait fall through, drains its MMAs and loads, frees
// TMEM and returns.
#include <cuda.h>

#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"
#include "tc_gates.cuh"

namespace cpdr {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 512;

// Modes: bit 0 = pre-process (else forward), bit 1 = per-dim gate (KDA),
// whose gate is folded into operand tiles precomputed per chunk (tc_kda.cu);
// bit 2 = layout variants in the forward (grouped query heads, [dv, dk]
// states), kept out of the plain forward's code (measured 4% slower with
// them compiled in).  The per-dim modes always handle the variants.
// The backward adds two modes: MODE_REC (bit 3) is the pre-process S chain
// run over every fragment from its initial state, storing the state at each
// chunk start and each chunk's Delta (the forward recomputation the input
// gradients need); MODE_BWD (bit 4) runs the state-gradient chain of the
// chunk form in reverse chunk order with the forward's warp roles and
// stage layout (V's slots hold dO); MODE_BWD_ACC (bit 5) is its pass for a
// state's query heads past the first.
// MODE_FWD_G2 (bit 6) is the forward of grouped query heads two at a time:
// with an even group size G each chain emits two query heads' outputs (G/2
// chains per state head).
enum Mode { MODE_FWD = 0, MODE_PRE = 1, MODE_FWD_KDA = 2, MODE_PRE_KDA = 3, MODE_FWD_VAR = 4, MODE_REC = 9,
            MODE_REC_KDA = 11, MODE_BWD = 16, MODE_BWD_KDA = 18, MODE_BWD_ACC = 48, MODE_BWD_KDA_ACC = 50,
            MODE_FWD_G2 = 68 };
__host__ __device__ constexpr bool mode_fwd(int m) { return (m & 1) == 0; }
__host__ __device__ constexpr bool mode_kda(int m) { return (m & 2) != 0; }
__host__ __device__ constexpr bool mode_var(int m) { return (m & 4) != 0 || (m & 3) != 0; }
__host__ __device__ constexpr bool mode_rec(int m) { return (m & 8) != 0; }
__host__ __device__ constexpr bool mode_bwd(int m) { return (m & 16) != 0; }
// the backward's later query-head passes (grouped query heads): no end
// gradient, and the stored sums are added to the first pass's
__host__ __device__ constexpr bool mode_acc(int m) { return (m & 32) != 0; }
__host__ __device__ constexpr bool mode_g2(int m) { return (m & 64) != 0; }
enum Role { ROLE_S = 0, ROLE_M = 1 };

// Optional event trace (compile with -DCPDR_TRACE): CTA (0, 0) of each
// launch records SM clock stamps per role, chunk and event.
#ifdef CPDR_TRACE
__device__ unsigned long long g_cpdr_trace[3][8][64][16];
#define TR(role, chunk, ev)                                                                \
    do {                                                                                   \
        if (blockIdx.x == 0 && blockIdx.y == 0 && (threadIdx.x & 31) == 0 && (chunk) < 64) \
            g_cpdr_trace[(MODE & 1) * (1 + ROLE)][role][chunk][ev] = (unsigned long long)clock64(); \
    } while (0)
#else
#define TR(role, chunk, ev) \
    do {                    \
    } while (0)
#endif

// TMEM columns (128 lanes each).  fp32 accumulators: P = [K; Q] K^T, W^T,
// Delta^T (over U^T), O^T, P_S.  bf16 A operands of later products, two
// values per column: -S^T (SB), -Delta^T (DB, forward) and (Delta diag
// Gamma)^T (DGB); the M chain's lo halves of -M^T and of (Delta diag Gamma)^T
// use the columns that P and DB occupy in the forward.
constexpr uint32_t TM_P = 0, TM_W = 64, TM_DL = 128, TM_O = 192, TM_PS = 256, TM_SB = 384, TM_DB = 448,
                   TM_DGB = 480;
constexpr uint32_t TM_SB_LO = 0, TM_DGB_LO = 448;
constexpr uint32_t TM_COLS = 512;
// The two-head forward: W^T and the two heads' Q K^T take columns 0..63 in
// turn, Delta^T 64..127, both heads' O^T 128..255 (head 0 first); the rest
// as above.
template <int MODE>
struct TMap {
    static constexpr uint32_t P = mode_g2(MODE) ? 0u : TM_P, W = mode_g2(MODE) ? 0u : TM_W,
                              DL = mode_g2(MODE) ? 64u : TM_DL, O = mode_g2(MODE) ? 128u : TM_O;
};

// mbarrier indices
enum Bar {
    B_FULL0, B_FULL1, B_FULL2, B_EMPTY0, B_EMPTY1, B_EMPTY2, B_PFULL, B_PFREE, B_WFULL, B_WREADY, B_WBFREE,
    B_UFULL, B_DLFULL, B_DLREADY, B_PSFULL, B_OFULL, B_OFREE, B_QREADY0, B_QREADY1, B_MREADY, B_MFREE,
    B_GATE0, B_GATE1, B_GATE2, B_GATE3, B_GATE4, B_DRAIN, B_DRAIN2, NBARS
};
constexpr int kMaxGateSlots = 5;
constexpr int kStateBar = 1;   // named barrier of the 8 state warps

struct Params {
    const cpdr_fragment *frags;
    const int32_t *items;
    const int32_t *chunk0;    // first global chunk of each fragment (WY tile order)
    const uint8_t *wy;        // WY tiles: [chunk][head][T', hi(T''), lo(T'')]
    const uint8_t *kda_qp;    // per-dim gate, grouped query heads: Qg and P of query heads 1 .. G-1
    const float *g;
    const float *S_init;
    __nv_bfloat16 *o;
    float *final_state;
    float *S_ext;
    float *M;
    int32_t *status;
    int H;
    int Hq, G;                // query heads of q and o, query heads per state (Hq = G H)
    int vfirst;               // dk x dv states stored [dv][dk]
    float scale;
    // backward: per (chunk, head) unit u = global chunk * H + head
    float *st_S;              // MODE_REC: S at each chunk start; MODE_BWD (main): dS after each chunk; [u][dk][dv]
    float *st_D;              // MODE_REC: Delta; MODE_BWD (main): dDelta; [u][64][dv]
    const float *dht;         // MODE_BWD: gradient of the final states [N][H][dk][dv] (nullable)
    const float *dS_end;      // MODE_BWD main: gradient at the end of continuing fragments [R*B][H][dk][dv]
    int bwd_pre;              // MODE_BWD: 1 = backward pre-process (dS at the fragment start into S_ext)
    int bwd_gq;               // MODE_BWD, grouped query heads: this pass's query head of each state
                              // (q and dO of head h G + bwd_gq); passes past the first start from
                              // zero and add their dS' / dDelta / dS_ext into the first pass's
};

// Shared-memory carve-up (byte offsets from a 1024-aligned base).
//   stage ring: K (and Q, V) tiles as two 64-column swizzled atoms each, and
//   the chunk's two WY tiles t1, t2 (T', hi(T'') for roles S and forward;
//   hi(T''), lo(T'') for role M)
struct Lay {
    uint32_t nstage, stage_bytes, kc0, kc1, qc0, qc1, vc0, vc1, t1, t2, k_lbo, v_lbo, tx_bytes, wy_off;
    uint32_t ngate, gate_floats;
    uint32_t mask, wb, wb_lo, gates, bars, ctl, tslot, total;
    // per-dim gate: operand tiles of the stage (Kg is kc0), the chunk decay,
    // the masked intra-chunk product, and the bulk copies from the unit
    uint32_t kgam, kglo, kgamlo, gcv, pt, gcs;
    uint32_t ncp, cp_src[3], cp_dst[3], cp_len[3];
};

__host__ __device__ constexpr Lay make_lay(int mode, int role) {
    Lay L{};
    if (mode_kda(mode)) {
        // stage images copied from the unit (offsets as in cpdr_internal.hpp)
        const uint32_t tp = 0, thi = (uint32_t)kWyTileBytes, tlo = 2 * (uint32_t)kWyTileBytes;
        const uint32_t gc = (uint32_t)kKdaOffGC, qg = (uint32_t)kKdaOffQg;
        if (mode_fwd(mode)) {
            L.t1 = 0; L.gcv = 8192; L.kc0 = 9216; L.kgam = 25600; L.qc0 = 41984; L.pt = 58368;
            L.vc0 = 66560; L.vc1 = 74752; L.stage_bytes = 82944;
            L.ncp = 3;
            L.cp_src[0] = tp; L.cp_dst[0] = L.t1; L.cp_len[0] = 8192;
            L.cp_src[1] = gc; L.cp_dst[1] = L.gcv; L.cp_len[1] = (uint32_t)(kKdaOffKgLo - kKdaOffGC);
            L.cp_src[2] = qg; L.cp_dst[2] = L.qc0; L.cp_len[2] = (uint32_t)(kKdaUnitBytes - kKdaOffQg);
            L.nstage = 2;
        } else if (role == ROLE_S) {
            L.t1 = 0; L.gcv = 8192; L.kc0 = 9216; L.kgam = 25600; L.vc0 = 41984; L.vc1 = 50176;
            L.stage_bytes = 58368;
            L.ncp = 2;
            L.cp_src[0] = tp; L.cp_dst[0] = L.t1; L.cp_len[0] = 8192;
            L.cp_src[1] = gc; L.cp_dst[1] = L.gcv; L.cp_len[1] = (uint32_t)(kKdaOffKgLo - kKdaOffGC);
            L.nstage = 3;
        } else {
            L.t1 = 0; L.t2 = 8192; L.gcv = 16384; L.kc0 = 17408; L.kgam = 33792; L.kglo = 50176;
            L.kgamlo = 66560; L.stage_bytes = 82944;
            L.ncp = 1;
            L.cp_src[0] = thi; L.cp_dst[0] = 0; L.cp_len[0] = (uint32_t)(kKdaOffQg - kWyTileBytes);
            L.nstage = 2;
            (void)tlo;
        }
        if (mode_fwd(mode) || role == ROLE_S) L.t2 = L.t1;   // T'' = T' (gamma is in the tiles)
        L.kc1 = L.kc0 + 8192; L.qc1 = L.qc0 + 8192; L.k_lbo = 8192; L.v_lbo = 8192; L.wy_off = 0;
        L.tx_bytes = L.stage_bytes;
        L.ngate = L.nstage + 2;
        L.gate_floats = 0;
        const bool split = !mode_fwd(mode) && role == ROLE_M;
        uint32_t o = L.nstage * L.stage_bytes;
        L.mask = o;
        L.wb = o; o += 16384;
        L.wb_lo = o; o += (split ? 16384 : 0);
        L.gates = o;
        L.gcs = o; o += 512;   // the state warps' copy of the chunk decay
        L.bars = o; o += NBARS * 8;
        L.ctl = o; o += 16;
        L.tslot = o; o += 16;
        L.total = o;
        return L;
    }
    if (mode_g2(mode)) {
        // per 64-column atom K | Q (head 0) | Q (head 1): [K; Q0] and [Q0; Q1]
        // are the stacked A operands of the two heads' Q K^T, [Q0; Q1] the B
        // operand of both heads' output product
        L.stage_bytes = 81920; L.kc0 = 0; L.qc0 = 8192; L.kc1 = 24576; L.qc1 = 32768; L.vc0 = 49152; L.vc1 = 57344;
        L.t1 = 65536; L.t2 = 73728;
        L.k_lbo = 24576; L.v_lbo = 8192; L.wy_off = 0;
    } else if (mode_fwd(mode)) {
        L.stage_bytes = 65536; L.kc0 = 0; L.qc0 = 8192; L.kc1 = 16384; L.qc1 = 24576; L.vc0 = 32768; L.vc1 = 40960;
        L.t1 = 49152; L.t2 = 57344;
        L.k_lbo = 16384; L.v_lbo = 8192; L.wy_off = 0;
    } else if (role == ROLE_S) {
        L.stage_bytes = 49152; L.kc0 = 0; L.vc0 = 8192; L.kc1 = 16384; L.vc1 = 24576; L.qc0 = 0; L.qc1 = 0;
        L.t1 = 32768; L.t2 = 40960;
        L.k_lbo = 16384; L.v_lbo = 16384; L.wy_off = 0;
    } else {
        L.stage_bytes = 32768; L.kc0 = 0; L.kc1 = 8192; L.qc0 = 0; L.qc1 = 0; L.vc0 = 0; L.vc1 = 0;
        L.t1 = 16384; L.t2 = 24576;
        L.k_lbo = 8192; L.v_lbo = 0; L.wy_off = (uint32_t)kWyTileBytes;
    }
    L.tx_bytes = L.stage_bytes;
    // three stages: a chunk's loads start two chunks ahead (the two-head
    // forward: two, for the second Q tile)
    L.nstage = mode_g2(mode) ? 2 : 3;
    // gate slots: a slot is rewritten once the chunk NG before it is
    // finished, which the stage ring guarantees for NG = stages + 2
    L.ngate = L.nstage + 2;
    // forward: G, gamma, Gamma, e, f (64 each), gamma^C, exact flag;
    // pre-process: Gamma, gamma^C
    L.gate_floats = (mode_fwd(mode)) ? 5 * 64 + 4 : 64 + 4;
    const bool split = (!mode_fwd(mode) && role == ROLE_M);
    uint32_t o = L.nstage * L.stage_bytes;
    L.mask = o; o += (mode_g2(mode) ? 16384 : mode_fwd(mode) ? 8192 : 0);   // the two-head forward: two masks
    L.wb = o; o += 16384;
    L.wb_lo = o; o += (split ? 16384 : 0);
    L.gates = o; o += L.ngate * L.gate_floats * 4;
    o = (o + 15) & ~15u;
    L.bars = o; o += NBARS * 8;
    L.ctl = o; o += 16;
    L.tslot = o; o += 16;
    L.total = o;
    L.kgam = L.kc0;   // scalar gate: one K tile serves every product
    return L;
}

// Per-CTA runtime state (registers once every role function is inlined).
struct Run {
    uint8_t *base;
    uint64_t *bar;
    Ctl *ctl;
    uint32_t tmem;
    int n, nlast, h, chunk0;
    int hq;                   // query head (forward; == h without grouped query heads)
    int64_t tok0;
    int seg, seq, flags;
    const Params *p;
    // chunk processed at iteration t (the backward runs in reverse)
    __device__ __forceinline__ int cof(int t, bool rev) const { return rev ? n - 1 - t : t; }
};

// gate slot arrays
struct Gates {
    float *G, *gam, *Gam, *e, *f, *gC;   // gC[0] = gamma^C, gC[1] = 1 when the exponentials must be exact
};
template <int MODE, int ROLE>
__device__ __forceinline__ Gates gates_of(const Run &r, int slot) {
    constexpr Lay L = make_lay(MODE, ROLE);
    float *q = reinterpret_cast<float *>(r.base + L.gates) + slot * L.gate_floats;
    if (mode_fwd(MODE)) return Gates{q, q + 64, q + 128, q + 192, q + 256, q + 320};
    return Gates{nullptr, nullptr, q, nullptr, nullptr, q + 64};
}
template <int MODE, int ROLE>
__device__ __forceinline__ int gate_slot(int c) { return c % (int)make_lay(MODE, ROLE).ngate; }
template <int MODE, int ROLE>
__device__ __forceinline__ uint32_t gate_parity(int c) { return (uint32_t)(c / (int)make_lay(MODE, ROLE).ngate) & 1u; }

__device__ __forceinline__ int rows_of(const Run &r, int chunk) { return chunk == r.n - 1 ? r.nlast : C; }

// Warp-uniform bounded wait on barrier b of the CTA.
__device__ __forceinline__ bool warp_wait(const Run &r, int b, uint32_t parity, int site) {
    return warp_wait_all(&r.bar[b], parity, r.ctl, r.p->status, site);
}

// ------------------------------------------------------------------ bf16 row stores
__device__ __forceinline__ uint4 pack8(const float *x) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]); u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]); u.w = pack_bf16(x[6], x[7]);
    return u;
}
__device__ __forceinline__ uint4 pack8_residual(const float *x, uint4 hi) {
    const __nv_bfloat162 *hp = reinterpret_cast<const __nv_bfloat162 *>(&hi);
    float lo[8];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const float2 f2 = __bfloat1622float2(hp[e]);
        lo[2 * e] = x[2 * e] - f2.x;
        lo[2 * e + 1] = x[2 * e + 1] - f2.y;
    }
    return pack8(lo);
}
// NQ 16-byte chunks (8 values each) of one 128-byte row, starting at chunk q0;
// with `lo` also the bf16 residual x - bf16(x).
template <int NQ>
__device__ __forceinline__ void store_row(uint8_t *tile, uint8_t *lo, uint32_t row, int q0, const float *x) {
#pragma unroll
    for (int q = 0; q < NQ; q++) {
        const uint4 u = pack8(x + 8 * q);
        const uint32_t off = sw128(row, q0 + q);
        *reinterpret_cast<uint4 *>(tile + off) = u;
        if (lo) *reinterpret_cast<uint4 *>(lo + off) = pack8_residual(x + 8 * q, u);
    }
}

// Bulk (non-tensor) copy global -> shared, completing on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------ producer
template <int MODE, int ROLE>
__device__ __forceinline__ void run_producer(const Run &r, const CUtensorMap *tq, const CUtensorMap *tk,
                                             const CUtensorMap *tv) {
    constexpr Lay L = make_lay(MODE, ROLE);
    const int lane = threadIdx.x & 31;
    const int H = r.p->H;
    int issued[3] = {-1, -1, -1};
    constexpr bool REV = mode_bwd(MODE);
    // in-chunk gates of the chunk of iteration t (padded rows: 0) -> its gate slot
    auto produce_gates = [&](int t) {
        const int c = r.cof(t, REV);
        const int nv = rows_of(r, c);
        const int64_t tk0 = r.tok0 + (int64_t)c * C;
        const int i0 = 2 * lane, i1 = 2 * lane + 1;
        float g0 = 0.f, g1 = 0.f;
        if (i0 < nv) g0 = r.p->g[(tk0 + i0) * H + r.h] * kLog2e;
        if (i1 < nv) g1 = r.p->g[(tk0 + i1) * H + r.h] * kLog2e;
        const LaneGates lg = scan_gates(g0, g1);
        const Gates gs = gates_of<MODE, ROLE>(r, gate_slot<MODE, ROLE>(t));
        gs.Gam[i0] = exp2f(lg.GC - lg.G0);
        gs.Gam[i1] = exp2f(lg.GC - lg.G1);
        if (mode_fwd(MODE)) {
            gs.G[i0] = lg.G0; gs.G[i1] = lg.G1;
            gs.gam[i0] = exp2f(lg.G0); gs.gam[i1] = exp2f(lg.G1);
            gs.e[i0] = exp2f(lg.G0 - lg.Gr); gs.e[i1] = exp2f(lg.G1 - lg.Gr);
            gs.f[i0] = exp2f(lg.Gr - lg.G0); gs.f[i1] = exp2f(lg.Gr - lg.G1);
        }
        if (lane == 0) {
            gs.gC[0] = exp2f(lg.GC);
            gs.gC[1] = lg.exact ? 1.f : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_GATE0 + gate_slot<MODE, ROLE>(t)]);
    };
    constexpr bool KDA = mode_kda(MODE);
    if (!KDA) produce_gates(0);
    constexpr int NS = (int)L.nstage;
    for (int t = 0; t < r.n; t++) {
        const int s = t % NS;
        int ok = 1;
        if (lane == 0 && t >= NS) ok = mbar_wait(&r.bar[B_EMPTY0 + s], ((t / NS) - 1) & 1, r.ctl, r.p->status, 10);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        TR(0, t, 0);
        uint64_t *fb = &r.bar[B_FULL0 + s];
        const int cc = r.cof(t, REV);   // the chunk this stage holds
        const int tok = (int)(r.tok0 + (int64_t)cc * C);
        if (KDA) {
            if (lane == 0) {
                // the unit's operand images, and V
                uint8_t *st = r.base + s * L.stage_bytes;
                const size_t u = (size_t)(r.chunk0 + cc) * H + r.h;
                const uint8_t *unit = r.p->wy + u * kKdaUnitBytes;
                // the forward's Qg and P (the last copy) belong to the query
                // head: query heads past a state's first keep theirs after
                // the units
                const int gq = mode_bwd(MODE) ? r.p->bwd_gq : mode_fwd(MODE) ? r.hq - r.h * r.p->G : 0;
                const uint8_t *qp = gq == 0 ? unit + kKdaOffQg
                                            : r.p->kda_qp + (u * (r.p->G - 1) + (gq - 1)) * kKdaQpBytes;
                mbar_arrive_expect_tx(fb, L.tx_bytes);
#pragma unroll
                for (int i = 0; i < (int)L.ncp; i++)
                    bulk_load(st + L.cp_dst[i], (mode_fwd(MODE) && i == 2) ? qp : unit + L.cp_src[i], L.cp_len[i], fb);
                if (mode_fwd(MODE) || ROLE == ROLE_S) {   // V (the backward: dO)
                    const int hv = mode_bwd(MODE) ? r.h * r.p->G + r.p->bwd_gq : r.h;
                    tma_load_3d(st + L.vc0, tv, fb, 0, hv, tok);
                    tma_load_3d(st + L.vc1, tv, fb, 64, hv, tok);
                }
            }
            issued[s] = t;
            continue;
        }
        if (lane == 0) {
            uint8_t *st = r.base + s * L.stage_bytes;
            mbar_arrive_expect_tx(fb, L.tx_bytes);
            tma_load_3d(st + L.kc0, tk, fb, 0, r.h, tok);
            tma_load_3d(st + L.kc1, tk, fb, 64, r.h, tok);
            // the backward's q and dO (in V's slots) are the pass's query head's
            const int hb = mode_bwd(MODE) ? r.h * r.p->G + r.p->bwd_gq : r.h;
            if (mode_fwd(MODE)) {
                const int hq = mode_var(MODE) ? r.hq : hb;
                tma_load_3d(st + L.qc0, tq, fb, 0, hq, tok);
                tma_load_3d(st + L.qc1, tq, fb, 64, hq, tok);
                if (mode_g2(MODE)) {   // the second query head's rows right after the first's
                    tma_load_3d(st + L.qc0 + 8192, tq, fb, 0, hq + 1, tok);
                    tma_load_3d(st + L.qc1 + 8192, tq, fb, 64, hq + 1, tok);
                }
            }
            if (mode_fwd(MODE) || ROLE == ROLE_S) {
                tma_load_3d(st + L.vc0, tv, fb, 0, hb, tok);
                tma_load_3d(st + L.vc1, tv, fb, 64, hb, tok);
            }
            const uint8_t *src = r.p->wy + ((size_t)(r.chunk0 + cc) * H + r.h) * kWyUnitBytes + L.wy_off;
            bulk_load(st + L.t1, src, 2 * (uint32_t)kWyTileBytes, fb);
        }
        // gates one chunk ahead of the stage ring
        if (t + 1 < r.n) produce_gates(t + 1);
        issued[s] = t;
    }
    // drain: every issued load must have landed before the CTA exits
    if (lane == 0) {
        Ctl local;
        local.abort = 0;
        for (int s = 0; s < NS; s++)
            if (issued[s] >= 0) mbar_wait(&r.bar[B_FULL0 + s], (issued[s] / NS) & 1, &local, r.p->status, 11);
    }
}

// ------------------------------------------------------------------ MMA issuer
// Descriptors are built once; a k-step adds (bytes >> 4) to the start field.
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return sdesc(addr, 16, 1024); }   // K-major SW128
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t lbo) { return sdesc(addr, lbo, 1024); }

// D(128 x N) (+)= A(128 x K, K-major, atom columns katom_a apart) * B(K-major rows = N)
template <int N, int K, bool NEG>
__device__ __forceinline__ void mma_kk(uint32_t d, uint64_t a, uint32_t katom_a, uint64_t b, uint32_t katom_b,
                                       bool acc) {
    constexpr uint32_t id = idesc_bf16(128, N, false, false, NEG);
#pragma unroll
    for (int k = 0; k < K / 16; k++) {
        const uint64_t ao = ((k & 3) * 32 + (k >> 2) * katom_a) >> 4, bo = ((k & 3) * 32 + (k >> 2) * katom_b) >> 4;
        mma_bf16(d, a + ao, b + bo, id, (acc || k > 0) ? 1u : 0u);
    }
}
// A K-major, B MN-major (K rows of 128 B, 2048 B per 16-row k-step)
template <int N, int K, bool NEG>
__device__ __forceinline__ void mma_kmn(uint32_t d, uint64_t a, uint32_t katom_a, uint64_t b, bool acc) {
    constexpr uint32_t id = idesc_bf16(128, N, false, true, NEG);
#pragma unroll
    for (int k = 0; k < K / 16; k++) {
        const uint64_t ao = ((k & 3) * 32 + (k >> 2) * katom_a) >> 4;
        mma_bf16(d, a + ao, b + (uint64_t)(k * 128), id, (acc || k > 0) ? 1u : 0u);
    }
}
// A MN-major (2048 B per k-step), B K-major
template <int N, int K>
__device__ __forceinline__ void mma_mnk(uint32_t d, uint64_t a, uint64_t b, uint32_t katom_b, bool acc) {
    constexpr uint32_t id = idesc_bf16(128, N, true, false, false);
#pragma unroll
    for (int k = 0; k < K / 16; k++) {
        const uint64_t bo = ((k & 3) * 32 + (k >> 2) * katom_b) >> 4;
        mma_bf16(d, a + (uint64_t)(k * 128), b + bo, id, (acc || k > 0) ? 1u : 0u);
    }
}

// A MN-major, B MN-major (2048 B per k-step each)
template <int N, int K>
__device__ __forceinline__ void mma_mnmn(uint32_t d, uint64_t a, uint64_t b, bool acc) {
    constexpr uint32_t id = idesc_bf16(128, N, true, true);
#pragma unroll
    for (int k = 0; k < K / 16; k++)
        mma_bf16(d, a + (uint64_t)(k * 128), b + (uint64_t)(k * 128), id, (acc || k > 0) ? 1u : 0u);
}

// D(128 x N) (+)= A(128 x K, in TMEM from column a) * B(MN-major, 2048 B per k-step)
template <int N, int K>
__device__ __forceinline__ void mma_tmn(uint32_t d, uint32_t a, uint64_t b, bool acc) {
    constexpr uint32_t id = idesc_bf16(128, N, false, true);
#pragma unroll
    for (int k = 0; k < K / 16; k++) mma_bf16_ts(d, a + 8 * k, b + (uint64_t)(k * 128), id, (acc || k > 0) ? 1u : 0u);
}
// D(128 x N) (+)= A(128 x K, in TMEM from column a) * B(K-major rows = N)
template <int N, int K>
__device__ __forceinline__ void mma_tk(uint32_t d, uint32_t a, uint64_t b, uint32_t katom_b, bool acc) {
    constexpr uint32_t id = idesc_bf16(128, N, false, false);
#pragma unroll
    for (int k = 0; k < K / 16; k++) {
        const uint64_t bo = ((k & 3) * 32 + (k >> 2) * katom_b) >> 4;
        mma_bf16_ts(d, a + 8 * k, b + bo, id, (acc || k > 0) ? 1u : 0u);
    }
}

// Shared-memory operand descriptors of one CTA (stage-0 addresses; stage s
// adds s * stage_bytes >> 4).
struct Descs {
    uint64_t stack0, kmn0, vmn0, q0, t10, t20, wb, wblo, mask;
    uint64_t kgam0, kglo0, kgamlo0, pt0;   // per-dim gate: P_S operands (hi, lo), W's lo operand, P
    uint64_t wbk, maskmn, qmn0;            // backward: W tile K-major, mask MN-major, gamma ⊙ Q MN-major
    uint64_t kgamk0, ptmn0;                // backward, per-dim gate: Kgam K-major, P MN-major
};
template <int MODE, int ROLE>
__device__ __forceinline__ Descs make_descs(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    const uint32_t b0 = smem_u32(r.base);
    Descs d;
    d.stack0 = kdesc(b0 + L.kc0);
    d.kmn0 = mndesc(b0 + L.kc0, L.k_lbo);
    d.vmn0 = mndesc(b0 + L.vc0, L.v_lbo);
    d.q0 = kdesc(b0 + L.qc0);
    d.t10 = kdesc(b0 + L.t1);
    d.t20 = kdesc(b0 + L.t2);
    d.wb = mndesc(b0 + L.wb, 16384);
    d.wblo = mndesc(b0 + L.wb_lo, 16384);
    d.mask = kdesc(b0 + L.mask);
    d.wbk = kdesc(b0 + L.wb);
    d.maskmn = mndesc(b0 + L.mask, 8192);
    d.qmn0 = mndesc(b0 + L.qc0, L.qc1 - L.qc0);
    if (mode_kda(MODE)) {
        d.kgam0 = mndesc(b0 + L.kgam, L.k_lbo);
        d.kglo0 = mndesc(b0 + L.kglo, L.k_lbo);
        d.kgamlo0 = mndesc(b0 + L.kgamlo, L.k_lbo);
        d.pt0 = kdesc(b0 + L.pt);
        d.kgamk0 = kdesc(b0 + L.kgam);
        d.ptmn0 = mndesc(b0 + L.pt, 8192);
    } else {
        d.kgam0 = d.kglo0 = d.kgamlo0 = d.pt0 = d.kgamk0 = d.ptmn0 = 0;
    }
    return d;
}
template <int MODE, int ROLE>
__device__ __forceinline__ uint64_t stg(uint64_t d, int t) {
    constexpr Lay L = make_lay(MODE, ROLE);
    return d + (uint64_t)((t % (int)L.nstage) * (L.stage_bytes >> 4));
}

// MMA warp: the products off the chain's critical path, as early as their
// inputs and TMEM columns allow -- chunk t's Q K^T (forward), W^T = K^T T''^T
// (hi + lo when split) and U^T = V^T T'^T.
template <int MODE, int ROLE>
__device__ __forceinline__ void run_mma(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool FWD = mode_fwd(MODE), SPLIT = (!mode_fwd(MODE) && ROLE == ROLE_M);
    constexpr bool HAS_U = FWD || ROLE == ROLE_S;
    constexpr bool KDA = mode_kda(MODE);
    constexpr int NS = (int)L.nstage;
    if ((threadIdx.x & 31) != 0) return;
    const uint32_t tm = r.tmem;
    int32_t *st = r.p->status;
    Ctl *ctl = r.ctl;
    const Descs d = make_descs<MODE, ROLE>(r);
    constexpr uint32_t KATOM = L.kc1 - L.kc0;
    // the backward's first products from dO (X1) are issued by the state warps
    constexpr bool MMA_U = HAS_U && !mode_bwd(MODE);
    if constexpr (mode_g2(MODE)) {
        // Two query heads per state: chunk t's W^T and U^T, then head 0's and
        // head 1's Q K^T in turn in the columns W^T used (each once its
        // previous reader is done), after chunk t-1's Delta product completed.
        // The mask-warp releases of the Q K^T columns alternate heads, so
        // head 0's is always phase parity 0 and head 1's parity 1.
        using T = TMap<MODE>;
        constexpr uint32_t QATOM = L.qc1 - L.qc0;
        for (int t = 0; t < r.n; t++) {
            if (!mbar_wait(&r.bar[B_FULL0 + t % NS], (t / NS) & 1, ctl, st, 20)) break;
            if (t >= 1 && !mbar_wait(&r.bar[B_WBFREE], (t - 1) & 1, ctl, st, 24)) break;
            if (t >= 1 && !mbar_wait(&r.bar[B_PFREE], 1, ctl, st, 22)) break;   // head 1's product of chunk t-1 read
            tc_fence_after();
            TR(1, t, 0);
            mma_mnk<64, 64>(tm + T::W, stg<MODE, ROLE>(d.kmn0, t), stg<MODE, ROLE>(d.t20, t), 8192, false);
            mma_commit(&r.bar[B_WFULL]);
            if (t >= 1 && !mbar_wait(&r.bar[B_DLREADY], (t - 1) & 1, ctl, st, 23)) break;
            tc_fence_after();
            mma_mnk<64, 64>(tm + T::DL, stg<MODE, ROLE>(d.vmn0, t), stg<MODE, ROLE>(d.t10, t), 8192, false);
            mma_commit(&r.bar[B_UFULL]);
            // head 0: P = [K; Q0] K^T, once the W epilogue has read W^T
            if (!mbar_wait(&r.bar[B_WREADY], t & 1, ctl, st, 21)) break;
            tc_fence_after();
            mma_kk<64, 128, false>(tm + T::P, stg<MODE, ROLE>(d.stack0, t), KATOM, stg<MODE, ROLE>(d.stack0, t),
                                   KATOM, false);
            mma_commit(&r.bar[B_PFULL]);
            // head 1: P = [Q0; Q1] K^T, once the mask warps have read head 0's
            if (!mbar_wait(&r.bar[B_PFREE], 0, ctl, st, 22)) break;
            tc_fence_after();
            mma_kk<64, 128, false>(tm + T::P, stg<MODE, ROLE>(d.q0, t), QATOM, stg<MODE, ROLE>(d.stack0, t), KATOM,
                                   false);
            mma_commit(&r.bar[B_PFULL]);
            mma_commit(&r.bar[B_EMPTY0 + t % NS]);   // this warp's reads of stage t
            TR(1, t, 1);
        }
        mma_commit(&r.bar[B_DRAIN]);
        Ctl local;
        local.abort = 0;
        mbar_wait(&r.bar[B_DRAIN], 0, &local, st, 30);
        return;
    }
    for (int t = 0; t < r.n; t++) {
        if (!mbar_wait(&r.bar[B_FULL0 + t % NS], (t / NS) & 1, ctl, st, 20)) break;
        // TMEM columns of W and P are free once chunk t-1's were read; the
        // products go into the tensor pipe after chunk t-1's Delta product
        // has completed (W behind it would delay the chain)
        if (t >= 1 && !mbar_wait(&r.bar[B_WREADY], (t - 1) & 1, ctl, st, 21)) break;
        if (t >= 1 && !mbar_wait(&r.bar[B_WBFREE], (t - 1) & 1, ctl, st, 24)) break;
        if (FWD && !KDA && t >= 1 && !mbar_wait(&r.bar[B_PFREE], (t - 1) & 1, ctl, st, 22)) break;
        tc_fence_after();
        TR(1, t, 0);
        if (FWD && !KDA) {   // P = [K; Q] K^T, rows 64..127 = Q K^T
            mma_kk<64, 128, false>(tm + TM_P, stg<MODE, ROLE>(d.stack0, t), KATOM, stg<MODE, ROLE>(d.stack0, t),
                                   KATOM, false);
            mma_commit(&r.bar[B_PFULL]);
        }
        const uint64_t tpp = SPLIT ? stg<MODE, ROLE>(d.t10, t) : stg<MODE, ROLE>(d.t20, t);
        mma_mnk<64, 64>(tm + TM_W, stg<MODE, ROLE>(d.kmn0, t), tpp, 8192, false);
        if (SPLIT) mma_mnk<64, 64>(tm + TM_W, stg<MODE, ROLE>(d.kmn0, t), stg<MODE, ROLE>(d.t20, t), 8192, true);
        // per-dim gate: the gated K tile is rounded too, W += lo(Kg) hi(T'')
        if (SPLIT && KDA) mma_mnk<64, 64>(tm + TM_W, stg<MODE, ROLE>(d.kglo0, t), tpp, 8192, true);
        mma_commit(&r.bar[B_WFULL]);
        if (MMA_U) {
            // the Delta accumulator is free once chunk t-1's Delta was read;
            // in the pre-process U goes in after chunk t-1's P_S has
            // completed; the forward issues it as soon as the Delta tile is
            // free (measured 2% faster A/B: it then completes during the
            // state update instead of after it)
            if (t >= 1 && !mbar_wait(&r.bar[B_DLREADY], (t - 1) & 1, ctl, st, 23)) break;
            if (!FWD && t >= 1 && !mbar_wait(&r.bar[B_PSFULL], (t - 1) & 1, ctl, st, 25)) break;
            tc_fence_after();
            mma_mnk<64, 64>(tm + TM_DL, stg<MODE, ROLE>(d.vmn0, t), stg<MODE, ROLE>(d.t10, t), 8192, false);
            mma_commit(&r.bar[B_UFULL]);
        }
        mma_commit(&r.bar[B_EMPTY0 + t % NS]);   // this warp's reads of stage t
        TR(1, t, 1);
    }
    // drain every MMA this thread issued
    mma_commit(&r.bar[B_DRAIN]);
    Ctl local;
    local.abort = 0;
    mbar_wait(&r.bar[B_DRAIN], 0, &local, st, 30);
}

// ------------------------------------------------------------------ mask warps (forward)
template <int MODE, int ROLE>
__device__ __forceinline__ void run_mask(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (mode_kda(MODE)) {
        // per-dim gate: gamma ⊙ Q and the masked product arrive with the
        // stage; release them chunk by chunk, one chunk ahead of the issuer
        constexpr int NS = (int)L.nstage;
        for (int ch = 0; ch < r.n; ch++) {
            if (ch >= 1 && !warp_wait(r, B_MFREE, (ch - 1) & 1, 53)) return;
            if (!warp_wait(r, B_FULL0 + ch % NS, (ch / NS) & 1, 54)) return;
            if (mode_bwd(MODE)) {
                // backward: the output scale into q 2^G and P (both multiply
                // dO), rows past the chunk's end zero (dO there belongs to the
                // next fragment)
                const int i = 32 * (w - 2) + lane;
                const float rs = i < rows_of(r, r.cof(ch, true)) ? r.p->scale : 0.f;
                const __nv_bfloat162 g2 = __float2bfloat162_rn(rs);
                uint8_t *stb = r.base + (ch % NS) * L.stage_bytes;
#pragma unroll
                for (int a = 0; a < 3; a++) {
                    uint8_t *tile = stb + (a == 0 ? L.qc0 : a == 1 ? L.qc1 : L.pt);
#pragma unroll
                    for (int c = 0; c < 8; c++) {
                        uint4 u = *reinterpret_cast<uint4 *>(tile + sw128(i, c));
                        __nv_bfloat162 *hh = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
                        for (int e = 0; e < 4; e++) hh[e] = __hmul2(hh[e], g2);
                        *reinterpret_cast<uint4 *>(tile + sw128(i, c)) = u;
                    }
                }
                fence_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&r.bar[B_QREADY0 + (ch & 1)]);
                mbar_arrive(&r.bar[B_MREADY]);
            }
        }
        return;
    }
    const int i = 32 * (w - 2) + lane;   // row of Q K^T (TMEM lane 64 + i)
    constexpr bool BWD = mode_bwd(MODE);
    if constexpr (mode_g2(MODE)) {
        // Two query heads: head 0's mask from the first Q K^T; once the second
        // product (which reads head 0's Q rows unscaled) has completed, both
        // heads' Q rows scaled by gamma_i in place, then head 1's mask.
        for (int ch = 0; ch < r.n; ch++) {
            if (!warp_wait(r, B_GATE0 + gate_slot<MODE, ROLE>(ch), gate_parity<MODE, ROLE>(ch), 50)) return;
            const Gates gs = gates_of<MODE, ROLE>(r, gate_slot<MODE, ROLE>(ch));
            const float Gi = gs.G[i], ei = gs.e[i];
            const bool exact = gs.gC[1] != 0.f;
#pragma unroll 1
            for (int hh = 0; hh < 2; hh++) {
                if (w == 2) TR(4, ch, hh);
                if (!warp_wait(r, B_PFULL, (uint32_t)hh, 51)) return;
                tc_fence_after();
                if (hh == 1) {
                    uint8_t *st = r.base + (ch % (int)L.nstage) * L.stage_bytes;
                    const __nv_bfloat162 g2 = __float2bfloat162_rn(gs.gam[i]);
#pragma unroll
                    for (int a = 0; a < 4; a++) {
                        uint8_t *tile = st + ((a & 1) ? L.qc1 : L.qc0) + (a >> 1) * 8192;
#pragma unroll
                        for (int c = 0; c < 8; c++) {
                            uint4 u = *reinterpret_cast<uint4 *>(tile + sw128(i, c));
                            __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
                            for (int e = 0; e < 4; e++) h[e] = __hmul2(h[e], g2);
                            *reinterpret_cast<uint4 *>(tile + sw128(i, c)) = u;
                        }
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&r.bar[B_QREADY0 + (ch & 1)]);
                }
                float m[64];
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    float v[32];
                    tmem_ld32(r.tmem + ((uint32_t)(64 + 32 * (w - 2)) << 16) + TMap<MODE>::P + 32 * half, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q4 = 0; q4 < 8; q4++) {
                        const int j0 = 32 * half + 4 * q4;
                        const float4 f4 = *reinterpret_cast<const float4 *>(gs.f + j0);
                        const float fv[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            const float x = v[4 * q4 + u];
                            const float val = exact ? x * exp2f(Gi - gs.G[j0 + u]) : x * ei * fv[u];
                            m[j0 + u] = (j0 + u <= i) ? val : 0.f;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&r.bar[B_PFREE]);
                // the previous chunk's masks must have been consumed
                if (hh == 0 && ch >= 1 && !warp_wait(r, B_MFREE, (ch - 1) & 1, 52)) return;
                store_row<8>(r.base + L.mask + 8192 * hh, nullptr, i, 0, m);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.bar[B_MREADY]);
            if (w == 2) TR(4, ch, 2);
        }
        return;
    }
    for (int ch = 0; ch < r.n; ch++) {
        if (!warp_wait(r, B_GATE0 + gate_slot<MODE, ROLE>(ch), gate_parity<MODE, ROLE>(ch), 50)) return;
        const Gates gs = gates_of<MODE, ROLE>(r, gate_slot<MODE, ROLE>(ch));
        // backward: the output scale goes into gamma ⊙ Q and the mask (both
        // multiply dO), and rows past the chunk's end are zero (dO there
        // belongs to the next fragment)
        const float rs = BWD ? (i < rows_of(r, r.cof(ch, true)) ? r.p->scale : 0.f) : 1.f;
        if (w == 2) TR(4, ch, 0);
        if (!warp_wait(r, B_PFULL, ch & 1, 51)) return;
        if (w == 2) TR(4, ch, 1);
        tc_fence_after();
        // Q K^T has been computed (first: the O product waits for it): scale
        // row i of this chunk's Q tile by gamma_i in place, so that
        // S^T (gamma ⊙ Q)^T and Delta^T mask^T accumulate into one TMEM tile
        {
            uint8_t *st = r.base + (ch % (int)L.nstage) * L.stage_bytes;
            const __nv_bfloat162 g2 = __float2bfloat162_rn(rs * gs.gam[i]);
#pragma unroll
            for (int a = 0; a < 2; a++) {
                uint8_t *tile = st + (a ? L.qc1 : L.qc0);
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    uint4 u = *reinterpret_cast<uint4 *>(tile + sw128(i, c));
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
                    for (int e = 0; e < 4; e++) h[e] = __hmul2(h[e], g2);
                    *reinterpret_cast<uint4 *>(tile + sw128(i, c)) = u;
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.bar[B_QREADY0 + (ch & 1)]);
        }
        const float Gi = gs.G[i], ei = gs.e[i];
        const bool exact = gs.gC[1] != 0.f;
        float m[64];
#pragma unroll
        for (int half = 0; half < 2; half++) {
            float v[32];
            tmem_ld32(r.tmem + ((uint32_t)(64 + 32 * (w - 2)) << 16) + TM_P + 32 * half, v);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 8; q4++) {
                const int j0 = 32 * half + 4 * q4;
                const float4 f4 = *reinterpret_cast<const float4 *>(gs.f + j0);
                const float fv[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const float x = v[4 * q4 + u];
                    const float val = exact ? x * exp2f(Gi - gs.G[j0 + u]) : x * ei * fv[u];
                    m[j0 + u] = (j0 + u <= i) ? rs * val : 0.f;
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_PFREE]);
        // the previous mask must have been consumed before this one is written
        if (ch >= 1 && !warp_wait(r, B_MFREE, (ch - 1) & 1, 52)) return;
        store_row<8>(r.base + L.mask, nullptr, i, 0, m);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_MREADY]);
        if (w == 2) TR(4, ch, 2);
    }
}

// ------------------------------------------------------------------ W and O epilogue warps
// W epilogue: W^T (TMEM lanes = dk) -> bf16 MN-major B tile of the Delta
// product (hi/lo when split).  O epilogue (forward): o = scale (gamma_i O1 +
// O2) for the 64 tokens of a chunk, TMEM lane = value dim; O1 + O2 arrive
// as one accumulator (the gamma_i row scale is folded into Q).  Per chunk t the
// warps handle W of chunk t+1 first (it gates the next Delta product), then O
// of chunk t.
template <int MODE, int ROLE>
__device__ __forceinline__ void run_wepi(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool FWD = mode_fwd(MODE), SPLIT = (!mode_fwd(MODE) && ROLE == ROLE_M);
    const Params &p = *r.p;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = w & 3, row = 32 * q + lane;
    const uint32_t lane_base = r.tmem + ((uint32_t)(32 * q) << 16);
    auto w_epilogue = [&](int t) -> bool {
        if (!warp_wait(r, B_WFULL, t & 1, 40)) return false;
        if (w == 4) TR(2, t, 0);
        tc_fence_after();
        float v0[32], v1[32];
        tmem_ld32(lane_base + TMap<MODE>::W, v0);
        tmem_ld32(lane_base + TMap<MODE>::W + 32, v1);
        tmem_ld_wait();
        tc_fence_before();
        // the previous chunk's Delta product must have read the tile
        if (t >= 1 && !warp_wait(r, B_WBFREE, (t - 1) & 1, 41)) return false;
        store_row<4>(r.base + L.wb, SPLIT ? r.base + L.wb_lo : nullptr, row, 0, v0);
        store_row<4>(r.base + L.wb, SPLIT ? r.base + L.wb_lo : nullptr, row, 4, v1);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_WREADY]);
        if (w == 4) TR(2, t, 1);
        return true;
    };
    if (!w_epilogue(0)) return;
    for (int t = 0; t < r.n; t++) {
        if (t + 1 < r.n && !w_epilogue(t + 1)) return;
        if (FWD && !mode_bwd(MODE)) {
            if (!warp_wait(r, B_OFULL, t & 1, 43)) return;
            if (w == 4) TR(2, t, 3);
            tc_fence_after();
            const int nv = rows_of(r, t);
            const int Hq = mode_var(MODE) ? p.Hq : p.H, hq = mode_var(MODE) ? r.hq : r.h;
            const int64_t ostride = (int64_t)Hq * D;
            __nv_bfloat16 *op = p.o + ((r.tok0 + (int64_t)t * C) * Hq + hq) * D + row;
            const float sc = -p.scale;   // the accumulator holds -O^T
            if constexpr (mode_g2(MODE)) {
                // both query heads (hq, hq + 1): head 0 read and stored, then
                // head 1 read, the accumulator released, head 1 stored (one
                // head's outputs in registers at a time)
#pragma unroll 1
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t pk[32];
#pragma unroll
                    for (int piece = 0; piece < 4; piece++) {   // 16 columns at a time
                        float a[16];
                        tmem_ld16(lane_base + TMap<MODE>::O + 64 * hh + 16 * piece, a);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; k++) pk[8 * piece + k] = pack_bf16(sc * a[2 * k], sc * a[2 * k + 1]);
                    }
                    if (hh == 1) {
                        if (w == 4) TR(2, t, 4);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&r.bar[B_OFREE]);
                    }
                    __nv_bfloat16 *q = op + hh * D;
#pragma unroll
                    for (int k = 0; k < 32; k++) {
                        if (2 * k < nv) *q = __ushort_as_bfloat16((unsigned short)(pk[k] & 0xffffu));
                        q += ostride;
                        if (2 * k + 1 < nv) *q = __ushort_as_bfloat16((unsigned short)(pk[k] >> 16));
                        q += ostride;
                    }
                }
                if (w == 4) TR(2, t, 2);
                continue;
            }
            float a[32], b[32];
            tmem_ld32(lane_base + TM_O, a);
            tmem_ld32(lane_base + TM_O + 32, b);
            tmem_ld_wait();
            if (w == 4) TR(2, t, 4);
            // the accumulator is in registers: release it before the stores
            // (an arrive after them would wait for the stores to complete)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.bar[B_OFREE]);
#pragma unroll
            for (int i = 0; i < 32; i++)
                if (i < nv) op[i * ostride] = __float2bfloat16_rn(sc * a[i]);
#pragma unroll
            for (int i = 0; i < 32; i++)
                if (32 + i < nv) op[(32 + i) * ostride] = __float2bfloat16_rn(sc * b[i]);
            if (w == 4) TR(2, t, 2);
        }
    }
}

// ------------------------------------------------------------------ state warps
// -x as bf16 pairs (and the residual pairs -x - bf16(-x) when lo != nullptr):
// column c of the pair array holds x[2c], x[2c+1].
template <int NC>
__device__ __forceinline__ void neg_pairs(const float *x, uint32_t (&hi)[NC], uint32_t *lo) {
#pragma unroll
    for (int c = 0; c < NC; c++) {
        const float a = -x[2 * c], b = -x[2 * c + 1];
        hi[c] = pack_bf16(a, b);
        if (lo) {
            const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi[c]));
            lo[c] = pack_bf16(a - h.x, b - h.y);
        }
    }
}

// Backward state warps: the state-gradient chain of the chunk form, chunks
// in reverse.  dS^T (rows = value dims) lives in their registers; per chunk,
// with the chunk's dO, Q, K, the WY product W and the masked product P (the
// reverse-mode derivative of the chunk equations of [FLA-CP] §2.2; the
// backward flow of §4):
//   dDelta^T = dO~^T P + Gamma ⊙ (dS'^T K^T)                    (X1 + Gamma X2)
//   dS^T     = gamma^C dS'^T + dO~^T (gamma ⊙ Q) - dDelta^T W   (X3 + X4)
// where dS' is the gradient after the chunk and dO~ = scale dO (the scale
// lives in the mask and in gamma ⊙ Q, which the mask warps prepare).  Lane 0
// of warp 8 issues X1, X2 and then X3, X4 right after the warps meet at their
// named barrier.  The main pass stores dS' and dDelta of every chunk; the
// pre-process keeps only the gradient at the fragment's start (S_ext).
template <int MODE, int ROLE>
__device__ __forceinline__ void run_state_bwd(const Run &r, float (&S)[64], int64_t sidx) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr int NS = (int)L.nstage;
    const Params &p = *r.p;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = w & 3, half = (w - 8) >> 2;
    const int row = 32 * q + lane;                       // TMEM lane: value dim
    const uint32_t tm = r.tmem;
    const uint32_t lane_base = tm + ((uint32_t)(32 * q) << 16);
    const bool issuer = (w == 8 && lane == 0);
    const int H = p.H;
    int32_t *st = p.status;
    Ctl *ctl = r.ctl;
    const Descs d = make_descs<MODE, ROLE>(r);
    constexpr uint32_t KATOM = L.kc1 - L.kc0;
    constexpr bool KDA = mode_kda(MODE);   // per-dim gate: Gamma lives in Kgam, gamma in q 2^G, the mask is P
    const bool main_pass = p.bwd_pre == 0;
    // dS^T[row][64 half .. 64 half + 63] as the bf16 A operand of X2
    auto put_grad = [&]() {
#pragma unroll
        for (int part = 0; part < 2; part++) {
            uint32_t hi[16];
#pragma unroll
            for (int c2 = 0; c2 < 16; c2++) hi[c2] = pack_bf16(S[32 * part + 2 * c2], S[32 * part + 2 * c2 + 1]);
            tmem_st16(lane_base + TM_SB + 32 * half + 16 * part, hi);
        }
        tmem_st_wait();
        tc_fence_before();
    };
    // the end gradient: dht where the sequence ends in this fragment; in the
    // main pass dS_end where the fragment continues into the next segment
    const float *src = nullptr;
    int64_t base = 0;
    bool tr = false;   // dht in the [dv][dk] layout
    constexpr bool accum = mode_acc(MODE);   // a later query head's pass: no end gradient, sums added
    if (accum) {
    } else if (r.flags & CPDR_FRAG_ENDS_SEQ) {
        if (p.dht) {
            src = p.dht;
            base = ((int64_t)r.seq * H + r.h) * D * D;
            tr = p.vfirst != 0;
        }
    } else if ((r.flags & CPDR_FRAG_CONT_NEXT) && main_pass) {
        src = p.dS_end;
        base = sidx;
    }
#pragma unroll
    for (int i = 0; i < 64; i++)
        S[i] = src ? src[base + (tr ? (int64_t)row * D + 64 * half + i : (int64_t)(64 * half + i) * D + row)] : 0.f;
    put_grad();
    int bad = named_bar_or(kStateBar, 256, 0);
    for (int t = 0; t < r.n && !bad; t++) {
        const int c = r.cof(t, true);
        const int nv = rows_of(r, c);
        const int64_t unit = (int64_t)(r.chunk0 + c) * H + r.h;
        if (main_pass) {   // dS' of the chunk, [dk][dv]
            float *dst = p.st_S + unit * D * D + row;
            if constexpr (accum) {
#pragma unroll
                for (int i = 0; i < 64; i++) dst[(int64_t)(64 * half + i) * D] += S[i];
            } else {
#pragma unroll
                for (int i = 0; i < 64; i++) dst[(int64_t)(64 * half + i) * D] = S[i];
            }
        }
        // ---- X1 = dO^T mask, X2 = dS'^T K^T  (per-dim gate: dO^T P, dS'^T Kgam^T)
        if (issuer) {
            if (mbar_wait(&r.bar[B_MREADY], t & 1, ctl, st, 70)) {
                tc_fence_after();
                mma_mnmn<64, 64>(tm + TM_DL, stg<MODE, ROLE>(d.vmn0, t),
                                 KDA ? stg<MODE, ROLE>(d.ptmn0, t) : d.maskmn, false);
                mma_commit(&r.bar[B_MFREE]);
                mma_tk<64, 128>(tm + TM_O, tm + TM_SB, stg<MODE, ROLE>(KDA ? d.kgamk0 : d.stack0, t), KATOM, false);
                mma_commit(&r.bar[B_DLFULL]);
            }
        }
        bool ok = KDA || warp_wait(r, B_GATE0 + gate_slot<MODE, ROLE>(t), gate_parity<MODE, ROLE>(t), 71);
        const Gates gs = gates_of<MODE, ROLE>(r, gate_slot<MODE, ROLE>(t));
        if (KDA && w == 8) {
            // the chunk's per-dim decay, kept past the stage's release
            const float4 g4 = reinterpret_cast<const float4 *>(r.base + (t % NS) * L.stage_bytes + L.gcv)[lane];
            reinterpret_cast<float4 *>(r.base + L.gcs)[lane] = g4;
        }
        if (ok) ok = warp_wait(r, B_DLFULL, t & 1, 72);
        if (ok) {
            tc_fence_after();
            float x1[32], x2[32];
            tmem_ld32(lane_base + TM_DL + 32 * half, x1);
            tmem_ld32(lane_base + TM_O + 32 * half, x2);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; jj++) {
                const int j = 32 * half + jj;
                x1[jj] = (j < nv) ? fmaf(KDA ? 1.f : gs.Gam[j], x2[jj], x1[jj]) : 0.f;
            }
            if (main_pass) {   // dDelta of the chunk, [64][dv]
                float *dst = p.st_D + unit * C * D + row;
                if constexpr (accum) {
#pragma unroll
                    for (int jj = 0; jj < 32; jj++) dst[(int64_t)(32 * half + jj) * D] += x1[jj];
                } else {
#pragma unroll
                    for (int jj = 0; jj < 32; jj++) dst[(int64_t)(32 * half + jj) * D] = x1[jj];
                }
            }
            uint32_t hi[16];   // -dDelta^T, the A operand of X4
            neg_pairs<16>(x1, hi, nullptr);
            tmem_st16(lane_base + TM_DGB + 16 * half, hi);
            tmem_st_wait();
            tc_fence_before();
        }
        if ((bad = named_bar_or(kStateBar, 256, ok ? 0 : 1))) break;
        // ---- X3 = dO^T (gamma ⊙ Q), X4 = (-dDelta^T) W, one accumulator
        if (issuer) {
            tc_fence_after();
            bool iok = mbar_wait(&r.bar[B_QREADY0 + (t & 1)], (t >> 1) & 1, ctl, st, 73);
            if (iok) iok = mbar_wait(&r.bar[B_WREADY], t & 1, ctl, st, 74);
            if (iok) {
                tc_fence_after();
                mma_mnmn<128, 64>(tm + TM_PS, stg<MODE, ROLE>(d.vmn0, t), stg<MODE, ROLE>(d.qmn0, t), false);
                mma_tk<128, 64>(tm + TM_PS, tm + TM_DGB, d.wbk, 8192, true);
                mma_commit(&r.bar[B_PSFULL]);
                mma_commit(&r.bar[B_WBFREE]);
                mma_commit(&r.bar[B_EMPTY0 + t % NS]);
            }
        }
        // ---- dS <- gamma^C dS' + X3 + X4  (per-dim gate: Diag(gamma^C), per key dim)
        ok = warp_wait(r, B_PSFULL, t & 1, 75);
        if (ok) {
            tc_fence_after();
            const float gC = KDA ? 0.f : gs.gC[0];
            const float *gcd = reinterpret_cast<const float *>(r.base + L.gcs) + 64 * half;
#pragma unroll
            for (int piece = 0; piece < 2; piece++) {
                float v[32];
                tmem_ld32(lane_base + TM_PS + 64 * half + 32 * piece, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++)
                    S[32 * piece + i] = fmaf(KDA ? gcd[32 * piece + i] : gC, S[32 * piece + i], v[i]);
            }
            put_grad();
        }
        bad = named_bar_or(kStateBar, 256, (ok && !ctl->abort) ? 0 : 1);
    }
    if (issuer) {   // drain every MMA this thread issued
        mma_commit(&r.bar[B_DRAIN2]);
        Ctl local;
        local.abort = 0;
        mbar_wait(&r.bar[B_DRAIN2], 0, &local, st, 76);
    }
    if (bad || main_pass) return;
    // the pre-process: the gradient at the fragment's start, [dk][dv]
    if constexpr (accum) {
#pragma unroll
        for (int i = 0; i < 64; i++) p.S_ext[sidx + (int64_t)(64 * half + i) * D + row] += S[i];
    } else {
#pragma unroll
        for (int i = 0; i < 64; i++) p.S_ext[sidx + (int64_t)(64 * half + i) * D + row] = S[i];
    }
}

// State warps (8-15): Delta epilogue and S update; lane 0 of warp 8 issues the
// chain's own products (Delta, O, P_S) right after the warps meet at a named
// barrier, so the critical path has no mbarrier hand-off to another warp.
template <int MODE, int ROLE>
__device__ __forceinline__ void run_state(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool FWD = mode_fwd(MODE), SPLIT = (!mode_fwd(MODE) && ROLE == ROLE_M);
    constexpr bool KDA = mode_kda(MODE);
    constexpr bool HAS_U = FWD || ROLE == ROLE_S;
    constexpr int NS = (int)L.nstage;
    const Params &p = *r.p;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = w & 3, half = (w - 8) >> 2;
    const int row = 32 * q + lane;                       // TMEM lane: value dim (or M column)
    const uint32_t tm = r.tmem;
    const uint32_t lane_base = tm + ((uint32_t)(32 * q) << 16);
    // the forward's products are issued by lane 0 of warp 8; in the
    // pre-process by warp 2, which joins the state warps' named barrier
    const bool issuer = FWD && (w == 8 && lane == 0);
    constexpr int kBarThreads = FWD ? 256 : 288;
    const int H = p.H;
    int32_t *st = p.status;
    Ctl *ctl = r.ctl;
    const Descs d = make_descs<MODE, ROLE>(r);
    constexpr uint32_t QATOM = L.qc1 - L.qc0;
    constexpr uint32_t tDL = TMap<MODE>::DL, tO = TMap<MODE>::O;
    constexpr int NO = mode_g2(MODE) ? 128 : 64;   // output columns: one or two query heads
    float S[64];
    const int64_t sidx = ((int64_t)r.seg * H + r.h) * D * D;
    if constexpr (mode_bwd(MODE)) {
        run_state_bwd<MODE, ROLE>(r, S, sidx);
        return;
    }
    constexpr bool REC = mode_rec(MODE);
    // -S^T[row][64 half .. 64 half + 63] as the bf16 A operand (hi, lo) of the
    // next Delta and O products
    auto put_state = [&]() {
#pragma unroll
        for (int part = 0; part < 2; part++) {
            uint32_t hi[16], lo[16];
            neg_pairs<16>(S + 32 * part, hi, SPLIT ? lo : nullptr);
            tmem_st16(lane_base + TM_SB + 32 * half + 16 * part, hi);
            if (SPLIT) tmem_st16(lane_base + TM_SB_LO + 32 * half + 16 * part, lo);
        }
        tmem_st_wait();
        tc_fence_before();
    };
    // initial state: S^T[row][64 half + i]
#pragma unroll
    for (int i = 0; i < 64; i++) {
        const int dk = 64 * half + i;
        float x = 0.f;
        if (SPLIT) x = (dk == row) ? 1.f : 0.f;
        else if ((FWD || REC) && (r.flags & CPDR_FRAG_CONT_PREV))
            x = p.S_init[sidx + ((mode_var(MODE) && p.vfirst) ? (int64_t)row * D + dk : (int64_t)dk * D + row)];
        S[i] = x;
    }
    put_state();
    int bad = named_bar_or(kStateBar, kBarThreads, 0);
    for (int ch = 0; ch < r.n && !bad; ch++) {
        const int64_t unit = (int64_t)(r.chunk0 + ch) * H + r.h;
        if (REC) {   // the state at the chunk's start, [dk][dv]
            float *dst = p.st_S + unit * D * D + row;
#pragma unroll
            for (int i = 0; i < 64; i++) dst[(int64_t)(64 * half + i) * D] = S[i];
        }
        // ---- Delta (and O) products of chunk ch
        if (issuer) {
            bool ok = mbar_wait(&r.bar[B_WREADY], ch & 1, ctl, st, 64);
            if (ok && HAS_U) ok = mbar_wait(&r.bar[B_UFULL], ch & 1, ctl, st, 65);
            if (ok) {
                tc_fence_after();
                TR(1, ch, 2);
                // Delta^T (+)= (-S^T) W^T
                if (!SPLIT) {
                    mma_tmn<64, 128>(tm + tDL, tm + TM_SB, d.wb, HAS_U);
                } else {
                    mma_tmn<64, 128>(tm + TM_DL, tm + TM_SB, d.wb, false);
                    mma_tmn<64, 128>(tm + TM_DL, tm + TM_SB_LO, d.wb, true);
                    mma_tmn<64, 128>(tm + TM_DL, tm + TM_SB, d.wblo, true);
                }
                mma_commit(&r.bar[B_WBFREE]);
                mma_commit(&r.bar[B_DLFULL]);   // the Delta epilogue need not wait for O1
            }
            if (ok && FWD) {   // -O^T = (-S^T) (gamma ⊙ Q)^T, before S is rewritten after P_S
                if (ch >= 1) ok = mbar_wait(&r.bar[B_OFREE], (ch - 1) & 1, ctl, st, 66);
                if (ok) ok = mbar_wait(&r.bar[B_QREADY0 + (ch & 1)], (ch >> 1) & 1, ctl, st, 67);
                if (ok) {
                    tc_fence_after();
                    // two heads: B = [gamma ⊙ Q0; gamma ⊙ Q1], N = 128
                    mma_tk<NO, 128>(tm + tO, tm + TM_SB, stg<MODE, ROLE>(d.q0, ch), QATOM, false);
                }
            }
            TR(1, ch, 3);
        }
        bool ok = KDA || warp_wait(r, B_GATE0 + gate_slot<MODE, ROLE>(ch), gate_parity<MODE, ROLE>(ch), 60);
        const Gates gs = gates_of<MODE, ROLE>(r, gate_slot<MODE, ROLE>(ch));
        // ---- Delta epilogue: tokens 32 half .. 32 half + 31 of Delta^T[row]
        if (w == 8) TR(3, ch, 0);
        if (ok) ok = warp_wait(r, B_DLFULL, ch & 1, 61);
        if (w == 8) TR(3, ch, 1);
        if (ok) {
            tc_fence_after();
            float v[32];
            tmem_ld32(lane_base + tDL + 32 * half, v);
            if (SPLIT) {   // the hi(-M^T) lo(W)^T half of the Delta product
#pragma unroll
                for (int part = 0; part < 2; part++) {
                    float u[16];
                    tmem_ld16(lane_base + TM_DL + 64 + 32 * half + 16 * part, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; i++) v[16 * part + i] += u[i];
                }
            }
            tmem_ld_wait();
            if (REC) {   // the chunk's Delta, [64][dv] (rows past the chunk's end: 0)
                const int nv = rows_of(r, ch);
                float *dst = p.st_D + unit * C * D + row;
#pragma unroll
                for (int jj = 0; jj < 32; jj++) dst[(int64_t)(32 * half + jj) * D] = (32 * half + jj < nv) ? v[jj] : 0.f;
            }
            if (FWD) {   // -Delta^T for the masked output product
                uint32_t d16[16];
                neg_pairs<16>(v, d16, nullptr);
                tmem_st16(lane_base + TM_DB + 16 * half, d16);
            }
            // (Delta diag Gamma)^T for P_S (negated here, so that the pair
            // conversion below stores it with a plus sign); per-dim gate:
            // Delta^T, Gamma being in the K operand
#pragma unroll
            for (int jj = 0; jj < 32; jj++) v[jj] = KDA ? -v[jj] : -(v[jj] * gs.Gam[32 * half + jj]);
            uint32_t hi[16], lo[16];
            neg_pairs<16>(v, hi, SPLIT ? lo : nullptr);
            tmem_st16(lane_base + TM_DGB + 16 * half, hi);
            if (SPLIT) tmem_st16(lane_base + TM_DGB_LO + 16 * half, lo);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (HAS_U && lane == 0) mbar_arrive(&r.bar[B_DLREADY]);   // the U product may reuse the columns
            if (KDA && w == 8) {
                // the chunk's per-dim decay, kept past the stage's release
                const float4 g4 = reinterpret_cast<const float4 *>(r.base + (ch % NS) * L.stage_bytes + L.gcv)[lane];
                reinterpret_cast<float4 *>(r.base + L.gcs)[lane] = g4;
            }
        }
        if (w == 8) TR(3, ch, 2);
        if ((bad = named_bar_or(kStateBar, kBarThreads, ok ? 0 : 1))) break;
        // ---- P_S (and the masked output product) of chunk ch
        if (issuer) {
            tc_fence_after();
            // P_S = (Delta diag Gamma)^T K  (per-dim gate: Delta^T Kgam)
            const uint64_t kps = KDA ? d.kgam0 : d.kmn0;   // scalar gate: one K tile for every product
            mma_tmn<128, 64>(tm + TM_PS, tm + TM_DGB, stg<MODE, ROLE>(kps, ch), false);
            if (SPLIT) mma_tmn<128, 64>(tm + TM_PS, tm + TM_DGB_LO, stg<MODE, ROLE>(kps, ch), true);
            if (SPLIT && KDA) mma_tmn<128, 64>(tm + TM_PS, tm + TM_DGB, stg<MODE, ROLE>(d.kgamlo0, ch), true);
            mma_commit(&r.bar[B_PSFULL]);
            TR(1, ch, 4);
            bool iok = true;
            if (FWD) {
                iok = mbar_wait(&r.bar[B_MREADY], ch & 1, ctl, st, 68);
                if (iok) {
                    tc_fence_after();
                    // -O^T += (-Delta^T) mask^T  (per-dim gate: the stage's P)
                    // two heads: B = [mask0; mask1], N = 128
                    mma_tk<NO, 64>(tm + tO, tm + TM_DB, KDA ? stg<MODE, ROLE>(d.pt0, ch) : d.mask, 8192, true);
                    mma_commit(&r.bar[B_OFULL]);
                    mma_commit(&r.bar[B_MFREE]);
                }
            }
            if (iok) mma_commit(&r.bar[B_EMPTY0 + ch % NS]);   // this thread's reads of stage ch
            TR(1, ch, 5);
        }
        // ---- state update: S <- gamma^C S + P_S
        ok = warp_wait(r, B_PSFULL, ch & 1, 62);
        if (w == 8) TR(3, ch, 3);
        if (ok) {
            tc_fence_after();
            const float gC = KDA ? 0.f : gs.gC[0];
            const float *gcd = reinterpret_cast<const float *>(r.base + L.gcs) + 64 * half;
#pragma unroll
            for (int piece = 0; piece < 2; piece++) {
                float v[32];
                tmem_ld32(lane_base + TM_PS + 64 * half + 32 * piece, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++)
                    S[32 * piece + i] = fmaf(KDA ? gcd[32 * piece + i] : gC, S[32 * piece + i], v[i]);
            }
            put_state();
        }
        if (w == 8) TR(3, ch, 4);
        bad = named_bar_or(kStateBar, kBarThreads, (ok && !ctl->abort) ? 0 : 1);
    }
    // drain every MMA the issuer issued
    if (issuer) {
        mma_commit(&r.bar[B_DRAIN2]);
        Ctl local;
        local.abort = 0;
        mbar_wait(&r.bar[B_DRAIN2], 0, &local, st, 69);
    }
    if (bad || REC) return;
    // outputs of the chain
    if (FWD) {
        // the first query head of a group writes the state's final value
        if ((r.flags & CPDR_FRAG_ENDS_SEQ) && p.final_state && (!mode_var(MODE) || r.hq % p.G == 0)) {
            const int64_t fidx = ((int64_t)r.seq * H + r.h) * D * D;
            if (mode_var(MODE) && p.vfirst) {   // [dv][dk]: this thread's row is contiguous
                float4 *dst = reinterpret_cast<float4 *>(p.final_state + fidx + (int64_t)row * D + 64 * half);
#pragma unroll
                for (int i = 0; i < 16; i++) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; i++) p.final_state[fidx + (int64_t)(64 * half + i) * D + row] = S[i];
            }
        }
    } else if (!SPLIT && p.vfirst) {   // S_ext [dv][dk]
        float4 *dst = reinterpret_cast<float4 *>(p.S_ext + sidx + (int64_t)row * D + 64 * half);
#pragma unroll
        for (int i = 0; i < 16; i++) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    } else {
        float *dst = SPLIT ? p.M : p.S_ext;
#pragma unroll
        for (int i = 0; i < 64; i++) dst[sidx + (int64_t)(64 * half + i) * D + row] = S[i];
    }
}

// Pre-process issuer (warp 2): issues the chain's Delta and P_S products
// right after the state warps meet at their named barrier, which it joins.
template <int MODE, int ROLE>
__device__ __forceinline__ void run_issuer(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool SPLIT = (!mode_fwd(MODE) && ROLE == ROLE_M);
    constexpr bool HAS_U = ROLE == ROLE_S;
    constexpr int NS = (int)L.nstage;
    const bool lead = (threadIdx.x & 31) == 0;
    const uint32_t tm = r.tmem;
    int32_t *st = r.p->status;
    Ctl *ctl = r.ctl;
    const Descs d = make_descs<MODE, ROLE>(r);
    int bad = named_bar_or(kStateBar, 288, 0);   // the initial state is in place
    for (int ch = 0; ch < r.n && !bad; ch++) {
        int ok = 1;
        if (lead) {
            ok = mbar_wait(&r.bar[B_WREADY], ch & 1, ctl, st, 64) ? 1 : 0;
            if (ok && HAS_U) ok = mbar_wait(&r.bar[B_UFULL], ch & 1, ctl, st, 65) ? 1 : 0;
            if (ok) {
                tc_fence_after();
                TR(1, ch, 2);
                // Delta^T (+)= (-S^T) W^T
                if (!SPLIT) {
                    mma_tmn<64, 128>(tm + TM_DL, tm + TM_SB, d.wb, HAS_U);
                } else {
                    // hi(-M^T) [hi(W) | lo(W)]^T as one N = 128 product (the
                    // two W images are one 64-column atom apart), its halves
                    // summed by the epilogue; lo(-M^T) hi(W)^T onto the first
                    mma_tmn<128, 128>(tm + TM_DL, tm + TM_SB, d.wb, false);
                    mma_tmn<64, 128>(tm + TM_DL, tm + TM_SB_LO, d.wb, true);
                }
                mma_commit(&r.bar[B_WBFREE]);
                mma_commit(&r.bar[B_DLFULL]);
            }
            TR(1, ch, 3);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // the state warps' Delta epilogue
        if ((bad = named_bar_or(kStateBar, 288, ok ? 0 : 1))) break;
        if (lead) {
            tc_fence_after();
            const uint64_t kps = mode_kda(MODE) ? d.kgam0 : d.kmn0;
            mma_tmn<128, 64>(tm + TM_PS, tm + TM_DGB, stg<MODE, ROLE>(kps, ch), false);
            if (SPLIT) mma_tmn<128, 64>(tm + TM_PS, tm + TM_DGB_LO, stg<MODE, ROLE>(kps, ch), true);
            if (SPLIT && mode_kda(MODE))
                mma_tmn<128, 64>(tm + TM_PS, tm + TM_DGB, stg<MODE, ROLE>(d.kgamlo0, ch), true);
            mma_commit(&r.bar[B_PSFULL]);
            mma_commit(&r.bar[B_EMPTY0 + ch % NS]);   // this thread's reads of stage ch
            TR(1, ch, 4);
        }
        __syncwarp();
        // the state warps' S update
        bad = named_bar_or(kStateBar, 288, ctl->abort ? 1 : 0);
    }
    if (lead) {
        mma_commit(&r.bar[B_DRAIN2]);
        Ctl local;
        local.abort = 0;
        mbar_wait(&r.bar[B_DRAIN2], 0, &local, st, 69);
    }
}

// ------------------------------------------------------------------ kernel
template <int MODE, int ROLE>
__device__ __forceinline__ void chain_body(uint8_t *base, const CUtensorMap *tq, const CUtensorMap *tk,
                                           const CUtensorMap *tv, const Params &p, int item) {
    constexpr Lay L = make_lay(MODE, ROLE);
    const int w = threadIdx.x >> 5;
    Run r;
    r.base = base;
    r.bar = reinterpret_cast<uint64_t *>(base + L.bars);
    r.ctl = reinterpret_cast<Ctl *>(base + L.ctl);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + L.tslot);
    const int fi = p.items[item];
    const cpdr_fragment f = p.frags[fi];
    r.tok0 = f.tok0;
    r.seg = f.seg;
    r.seq = f.seq;
    r.flags = f.flags;
    r.hq = blockIdx.y;
    // the forward's grid runs over query heads; the backward's over state heads
    r.h = (mode_var(MODE) && !mode_bwd(MODE)) ? r.hq / p.G : r.hq;
    if (mode_g2(MODE)) {   // G/2 chains per state head; chain j serves query heads h G + 2j and + 1
        const int pairs = p.G / 2;
        r.h = blockIdx.y / pairs;
        r.hq = r.h * p.G + 2 * (blockIdx.y % pairs);
    }
    r.n = (f.len + C - 1) / C;
    r.nlast = f.len - (r.n - 1) * C;
    r.chunk0 = p.chunk0[fi];
    r.p = &p;
    if (threadIdx.x == 0) {
        // arrival counts: PFREE / QREADY / MREADY 2 mask warps, WREADY / OFREE
        // 4 W/O-epilogue warps, DLREADY 8 state warps, EMPTY 2 MMA issuers
        uint32_t cnt[NBARS];
        for (int i = 0; i < NBARS; i++) cnt[i] = 1;
        cnt[B_PFREE] = 2;
        cnt[B_WREADY] = 4;
        cnt[B_DLREADY] = 8;
        cnt[B_EMPTY0] = cnt[B_EMPTY1] = cnt[B_EMPTY2] = 2;   // MMA warp + state issuer
        cnt[B_OFREE] = 4;
        cnt[B_MREADY] = 2;
        cnt[B_QREADY0] = cnt[B_QREADY1] = 2;
        for (int i = 0; i < NBARS; i++) mbar_init(&r.bar[i], cnt[i]);
        r.ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 0 && (threadIdx.x & 31) == 0) {
        if (!mode_kda(MODE)) tma_prefetch_desc(tk);
        if (mode_fwd(MODE) && !mode_kda(MODE)) tma_prefetch_desc(tq);
        if (mode_fwd(MODE) || ROLE == ROLE_S) tma_prefetch_desc(tv);
    }
    if (w == 1) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    r.tmem = *tmem_slot;
    if (w == 0) run_producer<MODE, ROLE>(r, tq, tk, tv);
    else if (w == 1) run_mma<MODE, ROLE>(r);
    else if (w < 4) {
        if (mode_fwd(MODE)) run_mask<MODE, ROLE>(r);
        else if (w == 2) run_issuer<MODE, ROLE>(r);
    }
    else if (w < 8) run_wepi<MODE, ROLE>(r);
    else run_state<MODE, ROLE>(r);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == 1) tmem_dealloc(r.tmem, TM_COLS);
}

template <int MODE, int ROLE>
__global__ void __launch_bounds__(NTHREADS, 1)
tc_chain_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic so that every
    // access through it stays a shared-space access
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    chain_body<MODE, ROLE>(base, &tq, &tk, &tv, p, blockIdx.x);
}

// The pre-process as one launch: blockIdx.z = 0 runs the transfer-matrix (M)
// chains, 1 the S chains.  Blocks are dispatched in grid order, so every M
// chain (the longer kind) starts before the S chains, which then fill the
// SMs the M chains leave: longest first within one launch.
template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
tc_pre_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
              const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    if (blockIdx.z == 0)
        chain_body<MODE, ROLE_M>(base, &tk, &tk, &tv, p, blockIdx.x);
    else
        chain_body<MODE, ROLE_S>(base, &tk, &tk, &tv, p, blockIdx.x);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [B*T, H, D] bf16 tensor, box {64, 1, 64}, 128-byte swizzle
bool make_tmap(CUtensorMap *m, const void *ptr, int64_t tokens, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kMaxSmem = 232448;   // 227 KiB opt-in per CTA
static_assert(make_lay(MODE_FWD, ROLE_S).total + 1024 <= kMaxSmem, "forward layout exceeds shared memory");
static_assert(make_lay(MODE_PRE, ROLE_S).total + 1024 <= kMaxSmem, "pre-process S layout exceeds shared memory");
static_assert(make_lay(MODE_PRE, ROLE_M).total + 1024 <= kMaxSmem, "pre-process M layout exceeds shared memory");
static_assert(make_lay(MODE_FWD_KDA, ROLE_S).total + 1024 <= kMaxSmem, "per-dim forward layout exceeds shared memory");
static_assert(make_lay(MODE_FWD_VAR, ROLE_S).total == make_lay(MODE_FWD, ROLE_S).total, "variant forward layout");
static_assert(make_lay(MODE_FWD_G2, ROLE_S).total + 1024 <= kMaxSmem && make_lay(MODE_FWD_G2, ROLE_S).ngate <= kMaxGateSlots,
              "two-head forward layout exceeds shared memory");
// the two-head forward's stacked operands: [K; Q0] and [Q0; Q1] contiguous per atom, the two masks adjacent
static_assert(make_lay(MODE_FWD_G2, ROLE_S).qc0 == make_lay(MODE_FWD_G2, ROLE_S).kc0 + 8192 &&
                  make_lay(MODE_FWD_G2, ROLE_S).kc1 - make_lay(MODE_FWD_G2, ROLE_S).kc0 ==
                      make_lay(MODE_FWD_G2, ROLE_S).qc1 - make_lay(MODE_FWD_G2, ROLE_S).qc0 &&
                  make_lay(MODE_FWD_G2, ROLE_S).qc0 + 16384 <= make_lay(MODE_FWD_G2, ROLE_S).kc1 &&
                  make_lay(MODE_FWD_G2, ROLE_S).qc1 + 16384 <= make_lay(MODE_FWD_G2, ROLE_S).vc0,
              "two-head forward stage layout");
// the M chain's fused Delta product reads hi(W) | lo(W) as one N = 128 operand (atom stride 16 KiB)
static_assert(make_lay(MODE_PRE, ROLE_M).wb_lo == make_lay(MODE_PRE, ROLE_M).wb + 16384 &&
                  make_lay(MODE_PRE_KDA, ROLE_M).wb_lo == make_lay(MODE_PRE_KDA, ROLE_M).wb + 16384,
              "W images of the M chain");
static_assert(make_lay(MODE_PRE_KDA, ROLE_S).total + 1024 <= kMaxSmem, "per-dim pre-process S layout too large");
static_assert(make_lay(MODE_PRE_KDA, ROLE_M).total + 1024 <= kMaxSmem, "per-dim pre-process M layout too large");
static_assert(make_lay(MODE_FWD_KDA, ROLE_S).tx_bytes < (1u << 20) && make_lay(MODE_PRE_KDA, ROLE_M).tx_bytes < (1u << 20),
              "stage bytes exceed the mbarrier transaction count");
static_assert(make_lay(MODE_FWD, ROLE_S).ngate <= kMaxGateSlots && make_lay(MODE_PRE, ROLE_M).ngate <= kMaxGateSlots,
              "gate slots exceed their barriers");
static_assert(make_lay(MODE_BWD, ROLE_S).total == make_lay(MODE_FWD, ROLE_S).total, "backward uses the forward layout");
static_assert(make_lay(MODE_BWD_ACC, ROLE_S).total == make_lay(MODE_BWD, ROLE_S).total, "the accumulating pass too");
static_assert(make_lay(MODE_REC, ROLE_S).total == make_lay(MODE_PRE, ROLE_S).total, "recompute uses the S layout");
static_assert(make_lay(MODE_REC_KDA, ROLE_S).total == make_lay(MODE_PRE_KDA, ROLE_S).total,
              "per-dim recompute uses the per-dim S layout");
static_assert(make_lay(MODE_BWD_KDA, ROLE_S).total == make_lay(MODE_FWD_KDA, ROLE_S).total &&
                  make_lay(MODE_BWD_KDA_ACC, ROLE_S).total == make_lay(MODE_FWD_KDA, ROLE_S).total,
              "per-dim backward uses the per-dim forward layout");

size_t smem_for(int mode, int role) { return make_lay(mode, role).total + 1024; }

template <int MODE>
int launch_pre_pair(const CUtensorMap &tk, const CUtensorMap &tv, const Params &prm, unsigned items, unsigned H,
                    cudaStream_t st) {
    const size_t sm = std::max(smem_for(MODE, ROLE_S), smem_for(MODE, ROLE_M));
    cudaError_t e = cudaFuncSetAttribute(tc_pre_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    tc_pre_kernel<MODE><<<dim3(items, H, 2), NTHREADS, sm, st>>>(tk, tv, prm);
    return (int)cudaGetLastError();
}

template <int MODE, int ROLE>
int launch_chain(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const Params &prm,
                 unsigned items, unsigned H, cudaStream_t st) {
    const size_t sm = smem_for(MODE, ROLE);
    cudaError_t e = cudaFuncSetAttribute(tc_chain_kernel<MODE, ROLE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sm);
    if (e != cudaSuccess) return (int)e;
    tc_chain_kernel<MODE, ROLE><<<dim3(items, H), NTHREADS, sm, st>>>(tq, tk, tv, prm);
    return (int)cudaGetLastError();
}

}  // namespace

#ifdef CPDR_TRACE
extern "C" int cpdr_debug_trace(unsigned long long *host, int n) {
    const int cap = (int)(sizeof(g_cpdr_trace) / 8);
    if (n > cap) n = cap;
    return (int)cudaMemcpyFromSymbol(host, g_cpdr_trace, (size_t)n * 8);
}
#endif

// bf16, d = 128 (both gates, grouped query heads and both state layouts)
bool tc_supported(const Plan &p) {
    return p.in_dtype == CPDR_DTYPE_BF16 && p.dk == 128 && p.dv == 128;
}

int launch_tc_pre(const cpdr_ctx *c, const void *k, const void *v, const float *g, const void *wy, float *S_ext,
                  float *M, void *stream) {
    const auto &p = c->plan;
    if (p.pre_items.empty()) return 0;
    CUtensorMap tk, tv;
    const int64_t tokens = (int64_t)p.B * p.T;
    const bool kda = p.gate_kind == CPDR_GATE_PER_DIM;   // K comes pre-gated in the units
    if (!make_tmap(&tk, kda ? v : k, tokens, p.H) || !make_tmap(&tv, v, tokens, p.H)) return (int)cudaErrorInvalidValue;
    Params prm{};
    prm.frags = c->dev.frags;
    prm.items = c->dev.pre_items;
    prm.chunk0 = c->dev.frag_chunk0;
    prm.wy = (const uint8_t *)wy;
    prm.g = g;
    prm.S_ext = S_ext;
    prm.M = M;
    prm.status = c->dev.status;
    prm.H = p.H;
    prm.Hq = p.H;
    prm.G = 1;
    prm.vfirst = p.vfirst;
    prm.scale = p.scale;
    // the transfer-matrix chains and the S chains in one launch, the longer
    // M chains dispatched first
    const unsigned items = (unsigned)p.pre_items.size(), H = (unsigned)p.H;
    return kda ? launch_pre_pair<MODE_PRE_KDA>(tk, tv, prm, items, H, (cudaStream_t)stream)
               : launch_pre_pair<MODE_PRE>(tk, tv, prm, items, H, (cudaStream_t)stream);
}

int launch_tc_fwd(const cpdr_ctx *c, const int32_t *items, int n_items, const void *q, const void *k, const void *v,
                  const float *g, const void *wy, const float *S_init, void *o, float *final_state, void *stream) {
    const auto &p = c->plan;
    if (n_items <= 0) return 0;
    CUtensorMap tq, tk, tv;
    const int64_t tokens = (int64_t)p.B * p.T;
    const bool kda = p.gate_kind == CPDR_GATE_PER_DIM;   // Q and K come pre-gated in the units
    if (!make_tmap(&tq, kda ? v : q, tokens, kda ? p.H : p.Hq) || !make_tmap(&tk, kda ? v : k, tokens, p.H) ||
        !make_tmap(&tv, v, tokens, p.H))
        return (int)cudaErrorInvalidValue;
    Params prm{};
    prm.frags = c->dev.frags;
    prm.items = items;
    prm.chunk0 = c->dev.frag_chunk0;
    prm.wy = (const uint8_t *)wy;
    prm.g = g;
    prm.S_init = S_init;
    prm.o = (__nv_bfloat16 *)o;
    prm.final_state = final_state;
    prm.status = c->dev.status;
    prm.H = p.H;
    prm.Hq = p.Hq;
    prm.G = p.G;
    prm.vfirst = p.vfirst;
    prm.scale = p.scale;
    if (kda) prm.kda_qp = (const uint8_t *)wy + p.wy_chunks.size() * (size_t)p.H * kKdaUnitBytes;
    // one chain per (fragment, query head): grouped query heads each run
    // their state head's chain, except with an even group size, where each
    // chain serves two query heads
    if (kda)
        return launch_chain<MODE_FWD_KDA, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.Hq,
                                                  (cudaStream_t)stream);
    // an even number of query heads per state: each chain emits two of them
    if (p.G % 2 == 0)
        return launch_chain<MODE_FWD_G2, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)(p.H * (p.G / 2)),
                                                 (cudaStream_t)stream);
    if (p.G > 1 || p.vfirst)
        return launch_chain<MODE_FWD_VAR, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.Hq,
                                                  (cudaStream_t)stream);
    return launch_chain<MODE_FWD, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.Hq, (cudaStream_t)stream);
}

}  // namespace cpdr

namespace cpdr {

// Backward, recomputation of the forward (MODE_REC): every fragment's S chain
// from its initial state (S_init where it continues a sequence), storing S at
// each chunk start (st_S, [unit][dk][dv]) and each chunk's Delta (st_D,
// [unit][64][dv]); unit = global chunk * H + head.
int launch_tc_rec(const cpdr_ctx *c, const void *k, const void *v, const float *g, const void *wy,
                  const float *S_init, float *st_S, float *st_D, void *stream) {
    const auto &p = c->plan;
    if (p.frags.empty()) return 0;
    CUtensorMap tk, tv;
    const int64_t tokens = (int64_t)p.B * p.T;
    if (!make_tmap(&tk, k, tokens, p.H) || !make_tmap(&tv, v, tokens, p.H)) return (int)cudaErrorInvalidValue;
    Params prm{};
    prm.frags = c->dev.frags;
    prm.items = c->dev.fwd_order;
    prm.chunk0 = c->dev.frag_chunk0;
    prm.wy = (const uint8_t *)wy;
    prm.g = g;
    prm.S_init = S_init;
    prm.status = c->dev.status;
    prm.H = p.H;
    prm.Hq = p.H;
    prm.G = 1;
    prm.scale = p.scale;
    prm.vfirst = p.vfirst;
    prm.st_S = st_S;
    prm.st_D = st_D;
    if (p.gate_kind == CPDR_GATE_PER_DIM)   // K comes pre-gated in the units
        return launch_chain<MODE_REC_KDA, ROLE_S>(tk, tk, tv, prm, (unsigned)p.frags.size(), (unsigned)p.H,
                                                  (cudaStream_t)stream);
    return launch_chain<MODE_REC, ROLE_S>(tk, tk, tv, prm, (unsigned)p.frags.size(), (unsigned)p.H,
                                          (cudaStream_t)stream);
}

// Backward, state-gradient chains (MODE_BWD) over `items`: pre = 1 writes the
// gradient at each fragment's start into dS_ext; pre = 0 stores dS after each
// chunk (st_dS, [unit][dk][dv]) and dDelta (st_dD, [unit][64][dv]).  With
// grouped query heads the chain is linear in its q / dO terms, so it runs
// once per query head of a state (gq = 0 .. G-1): the first pass starts
// from the end gradients and writes, the others start from zero and add.
int launch_tc_bwd_chain(const cpdr_ctx *c, const int32_t *items, int n_items, int pre, int gq, const void *q,
                        const void *k, const void *dout, const float *g, const void *wy, const float *dht,
                        const float *dS_end, float *dS_ext, float *st_dS, float *st_dD, void *stream) {
    const auto &p = c->plan;
    if (n_items <= 0) return 0;
    CUtensorMap tq, tk, tv;
    const int64_t tokens = (int64_t)p.B * p.T;
    if (!make_tmap(&tq, q, tokens, p.Hq) || !make_tmap(&tk, k, tokens, p.H) || !make_tmap(&tv, dout, tokens, p.Hq))
        return (int)cudaErrorInvalidValue;
    Params prm{};
    prm.frags = c->dev.frags;
    prm.items = items;
    prm.chunk0 = c->dev.frag_chunk0;
    prm.wy = (const uint8_t *)wy;
    prm.g = g;
    prm.S_ext = dS_ext;
    prm.status = c->dev.status;
    prm.H = p.H;
    prm.Hq = p.H;
    prm.G = 1;
    prm.scale = p.scale;
    prm.st_S = st_dS;
    prm.st_D = st_dD;
    prm.dht = dht;
    prm.dS_end = dS_end;
    prm.bwd_pre = pre;
    prm.G = p.G;
    prm.bwd_gq = gq;
    prm.vfirst = p.vfirst;
    if (p.gate_kind == CPDR_GATE_PER_DIM) {   // Q, K, P come pre-gated in the units
        prm.kda_qp = (const uint8_t *)wy + p.wy_chunks.size() * (size_t)p.H * kKdaUnitBytes;
        if (gq > 0)
            return launch_chain<MODE_BWD_KDA_ACC, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.H,
                                                          (cudaStream_t)stream);
        return launch_chain<MODE_BWD_KDA, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.H,
                                                  (cudaStream_t)stream);
    }
    if (gq > 0)
        return launch_chain<MODE_BWD_ACC, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.H,
                                                  (cudaStream_t)stream);
    return launch_chain<MODE_BWD, ROLE_S>(tq, tk, tv, prm, (unsigned)n_items, (unsigned)p.H, (cudaStream_t)stream);
}

}  // namespace cpdr
