// Tensor-core (tcgen05 / TMEM / TMA) kernels for the bf16, d = 128 path of
// the segmented delta-rule forward, scalar gate (GDN).
//
// One CTA runs one chain: a (fragment, head) pair, 64-token chunks in order.
// Per chunk, following the chunk form of the article "flash-linear-attention
// 上下文并行CP ..." ([FLA-CP] §2.2) in transposed storage (state rows = value
// dims, so every product has M = 128 on the tensor core):
//   P      = [K; Q] K^T                 (K K^T and Q K^T in one M=128 MMA)
//   A      = beta_i 2^(G_i - G_j) (K K^T)_ij, j < i          (SIMT)
//   T      = (I + A)^-1, T' = T diag(beta), T'' = T diag(beta gamma)   (SIMT, fp32)
//   W^T    = K^T T''^T,  U^T = V^T T'^T                      (MMA)
//   Delta^T= U^T - S^T W^T                                   (MMA, accumulate)
//   O^T    = S^T Q^T scaled by gamma_i + Delta^T mask^T,  mask_ij = (Q K^T)_ij 2^(G_i - G_j), j <= i
//   S^T   <- gamma^C S^T + (Delta diag(Gamma))^T K,  Gamma_j = 2^(G_C - G_j)
// The pre-process runs the same chain without outputs on the S columns
// (role S) and, in the same launch, the transfer-matrix chain
//   M <- M_[t] M,  M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W   ([FLA-CP] §2.2)
// (role M: U = 0, M_0 = I).  The M chain keeps fp32 accuracy, as the article
// requires: its accumulator lives in fp32 registers and every tensor-core
// operand derived from a rounded quantity (T'', W, M, Delta) is split into a
// bf16 hi/lo pair, so each product is hi*hi + lo*hi + hi*lo.
//
// Warp roles (16 warps): 0 TMA producer; 1 MMA issuer (+ TMEM owner);
// 2-3 causal mask (forward only); 4-7 gates, solve and the W epilogue;
// 8-15 state warps (Delta, S and O epilogues; the fp32 state lives in their
// registers, 64 values per thread).  Every wait is bounded: on expiry the
// kernel records a status code, raises an abort flag that makes every other
// wait fall through, drains its MMAs and loads, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"

namespace cpdr {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 512;
constexpr float kLog2e = 1.4426950408889634f;

enum Mode { MODE_FWD = 0, MODE_PRE = 1 };
enum Role { ROLE_S = 0, ROLE_M = 1 };

// TMEM columns (fp32, 128 lanes each)
constexpr uint32_t TM_P = 0, TM_W = 64, TM_DL = 128, TM_O1 = 192, TM_O2 = 256, TM_PS = 320;
constexpr uint32_t TM_COLS = 512;

// mbarrier indices
enum Bar {
    B_FULL0, B_FULL1, B_EMPTY0, B_EMPTY1, B_PFULL, B_PFREE, B_TREADY, B_TFREE, B_MREADY, B_MFREE,
    B_WFULL, B_WREADY, B_DLFULL, B_DLREADY, B_PSFULL, B_SREADY, B_OFULL, B_OFREE,
    B_GATE0, B_GATE1, B_GATE2, B_GATE3, B_WG, B_DRAIN, NBARS
};

struct Params {
    const cpdr_fragment *frags;
    const int32_t *items;
    const __nv_bfloat16 *beta;
    const float *g;
    const float *S_init;
    __nv_bfloat16 *o;
    float *final_state;
    float *S_ext;
    float *M;
    int32_t *status;
    int H;
    float scale;
};

// Shared-memory carve-up (byte offsets from a 1024-aligned base).
struct Lay {
    uint32_t stage_bytes, kc0, kc1, qc0, qc1, vc0, vc1, k_lbo, v_lbo, tx_bytes;
    uint32_t tp, tpp, tpp_lo, mask, wb, wb_lo, sb, sb_lo, db, dgb, dgb_lo, scr, tmp, gates, bars, total;
};

__host__ __device__ inline Lay make_lay(int mode, int role) {
    Lay L{};
    uint32_t o = 0;
    if (mode == MODE_FWD) {
        L.stage_bytes = 49152; L.kc0 = 0; L.qc0 = 8192; L.kc1 = 16384; L.qc1 = 24576; L.vc0 = 32768; L.vc1 = 40960;
        L.k_lbo = 16384; L.v_lbo = 8192; L.tx_bytes = 49152;
    } else if (role == ROLE_S) {
        L.stage_bytes = 32768; L.kc0 = 0; L.vc0 = 8192; L.kc1 = 16384; L.vc1 = 24576; L.qc0 = L.qc1 = 0;
        L.k_lbo = 16384; L.v_lbo = 16384; L.tx_bytes = 32768;
    } else {
        L.stage_bytes = 16384; L.kc0 = 0; L.kc1 = 8192; L.qc0 = L.qc1 = L.vc0 = L.vc1 = 0;
        L.k_lbo = 8192; L.v_lbo = 0; L.tx_bytes = 16384;
    }
    o = 2 * L.stage_bytes;
    const bool split = (mode == MODE_PRE && role == ROLE_M);
    L.tp = o; o += (split ? 0 : 8192);
    L.tpp = o; o += 8192;
    L.tpp_lo = o; o += (split ? 8192 : 0);
    L.mask = o; o += (mode == MODE_FWD ? 8192 : 0);
    L.wb = o; o += 16384;
    L.wb_lo = o; o += (split ? 16384 : 0);
    L.sb = o; o += 32768;
    L.sb_lo = o; o += (split ? 32768 : 0);
    L.db = o; o += (mode == MODE_FWD ? 16384 : 0);
    L.dgb = o; o += 16384;
    L.dgb_lo = o; o += (split ? 16384 : 0);
    L.scr = o; o += 64 * 65 * 4;              // solve scratch, fp32 [64][65]
    L.tmp = o; o += 48 * 16 * 4;              // solve temporary
    L.gates = o; o += 4 * (4 * 64 + 4) * 4;   // 4 slots: G, beta, gamma, Gamma, gamma^C
    o = (o + 15) & ~15u;
    L.bars = o; o += NBARS * 8 + 16 /*Ctl*/ + 16 /*TMEM base*/;
    L.total = o;
    return L;
}

// gate slot arrays
struct Gates {
    float *G, *beta, *gam, *Gam, *gC;
};
__device__ __forceinline__ Gates gates_of(uint8_t *base, const Lay &L, int slot) {
    float *p = reinterpret_cast<float *>(base + L.gates) + slot * (4 * 64 + 4);
    return Gates{p, p + 64, p + 128, p + 192, p + 256};
}

struct Ctx {
    uint8_t *base;
    uint64_t *bar;
    Ctl *ctl;
    uint32_t tmem;
    Lay L;
    int mode, role;
    int n;          // chunks
    int nlast;      // valid rows of the last chunk
    cpdr_fragment f;
    int h;
    const Params *p;
};

__device__ __forceinline__ uint32_t sa(const Ctx &c, uint32_t off) { return smem_u32(c.base + off); }

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast, then
// every lane performs its own (now immediate) acquire.
__device__ __forceinline__ bool warp_wait(const Ctx &c, int b, uint32_t parity, int site) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(&c.bar[b], parity, c.ctl, c.p->status, site) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(&c.bar[b], parity);
    return ok != 0;
}

// Bounded group barrier of the 4 solve warps (mbarrier with 4 arrivals).
__device__ __forceinline__ bool wg_sync(const Ctx &c, uint32_t &phase, int site) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&c.bar[B_WG]);
    const bool ok = warp_wait(c, B_WG, phase & 1, site);
    phase++;
    return ok;
}

__device__ __forceinline__ int rows_of(const Ctx &c, int chunk) { return chunk == c.n - 1 ? c.nlast : C; }

// ------------------------------------------------------------------ producer
__device__ void run_producer(const Ctx &c, const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv) {
    if ((threadIdx.x & 31) != 0) return;
    const Lay &L = c.L;
    int issued[2] = {-1, -1};
    for (int t = 0; t < c.n; t++) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait(&c.bar[B_EMPTY0 + s], ((t >> 1) - 1) & 1, c.ctl, c.p->status, 10)) break;
        uint8_t *st = c.base + s * L.stage_bytes;
        const int tok = (int)(c.f.tok0 + (int64_t)t * C);
        mbar_arrive_expect_tx(&c.bar[B_FULL0 + s], L.tx_bytes);
        tma_load_3d(st + L.kc0, tk, &c.bar[B_FULL0 + s], 0, c.h, tok);
        tma_load_3d(st + L.kc1, tk, &c.bar[B_FULL0 + s], 64, c.h, tok);
        if (c.mode == MODE_FWD) {
            tma_load_3d(st + L.qc0, tq, &c.bar[B_FULL0 + s], 0, c.h, tok);
            tma_load_3d(st + L.qc1, tq, &c.bar[B_FULL0 + s], 64, c.h, tok);
        }
        if (c.mode == MODE_FWD || c.role == ROLE_S) {
            tma_load_3d(st + L.vc0, tv, &c.bar[B_FULL0 + s], 0, c.h, tok);
            tma_load_3d(st + L.vc1, tv, &c.bar[B_FULL0 + s], 64, c.h, tok);
        }
        issued[s] = t;
    }
    // drain: every issued load must have landed before the CTA exits
    for (int s = 0; s < 2; s++)
        if (issued[s] >= 0) {
            Ctl tmp;
            tmp.abort = 0;
            mbar_wait(&c.bar[B_FULL0 + s], (issued[s] >> 1) & 1, &tmp, c.p->status, 11);
        }
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return sdesc(addr, 16, 1024); }       // K-major SW128
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t lbo) { return sdesc(addr, lbo, 1024); }

// D(128 x N) (+)= A(128 x K, K-major, atom columns at +katom) * B(K x N, K-major rows = N)
__device__ __forceinline__ void mma_kk(uint32_t d, uint32_t a, uint32_t katom_a, uint32_t b, uint32_t katom_b, int N,
                                       int K, bool neg, bool acc) {
    const uint32_t id = idesc_bf16(128, N, false, false, neg);
    for (int k = 0; k < K / 16; k++) {
        const uint32_t ao = (k & 3) * 32 + (k >> 2) * katom_a, bo = (k & 3) * 32 + (k >> 2) * katom_b;
        mma_bf16(d, kdesc(a + ao), kdesc(b + bo), id, (acc || k > 0) ? 1u : 0u);
    }
}
// A K-major, B MN-major (K rows of 128 B, N blocks at +lbo)
__device__ __forceinline__ void mma_kmn(uint32_t d, uint32_t a, uint32_t katom_a, uint32_t b, uint32_t lbo_b, int N,
                                        int K, bool neg, bool acc) {
    const uint32_t id = idesc_bf16(128, N, false, true, neg);
    for (int k = 0; k < K / 16; k++) {
        const uint32_t ao = (k & 3) * 32 + (k >> 2) * katom_a;
        mma_bf16(d, kdesc(a + ao), mndesc(b + k * 2048, lbo_b), id, (acc || k > 0) ? 1u : 0u);
    }
}
// A MN-major (M = 128 over blocks at +lbo_a), B K-major
__device__ __forceinline__ void mma_mnk(uint32_t d, uint32_t a, uint32_t lbo_a, uint32_t b, uint32_t katom_b, int N,
                                        int K, bool acc) {
    const uint32_t id = idesc_bf16(128, N, true, false, false);
    for (int k = 0; k < K / 16; k++) {
        const uint32_t bo = (k & 3) * 32 + (k >> 2) * katom_b;
        mma_bf16(d, mndesc(a + k * 2048, lbo_a), kdesc(b + bo), id, (acc || k > 0) ? 1u : 0u);
    }
}

__device__ void run_mma(const Ctx &c) {
    if ((threadIdx.x & 31) != 0) return;
    const Lay &L = c.L;
    const uint32_t tm = c.tmem;
    const bool fwd = c.mode == MODE_FWD, split = (c.mode == MODE_PRE && c.role == ROLE_M);
    const bool has_u = fwd || c.role == ROLE_S;
    int *st = c.p->status;
    Ctl *ctl = c.ctl;
    auto stage = [&](int t) { return sa(c, (t & 1) * L.stage_bytes); };
    // P = [K; Q] K^T  (rows 64..127 of the A tile are Q, V or unused)
    auto mma1 = [&](int t) {
        const uint32_t s0 = stage(t);
        mma_kk(tm + TM_P, s0 + L.kc0, L.kc1 - L.kc0, s0 + L.kc0, L.kc1 - L.kc0, 64, 128, false, false);
        mma_commit(&c.bar[B_PFULL]);
    };
    // W^T = K^T T''^T (hi and lo parts for the split chain), U^T = V^T T'^T
    auto emma = [&](int t) {
        const uint32_t s0 = stage(t);
        mma_mnk(tm + TM_W, s0 + L.kc0, L.k_lbo, sa(c, L.tpp), 8192, 64, 64, false);
        if (split) mma_mnk(tm + TM_W, s0 + L.kc0, L.k_lbo, sa(c, L.tpp_lo), 8192, 64, 64, true);
        mma_commit(&c.bar[B_WFULL]);
        if (has_u) mma_mnk(tm + TM_DL, s0 + L.vc0, L.v_lbo, sa(c, L.tp), 8192, 64, 64, false);
        mma_commit(&c.bar[B_TFREE]);
    };
    do {
        if (!mbar_wait(&c.bar[B_FULL0], 0, ctl, st, 20)) break;
        tc_fence_after();
        mma1(0);
        if (!mbar_wait(&c.bar[B_TREADY], 0, ctl, st, 21)) break;
        tc_fence_after();
        emma(0);
        for (int t = 0; t < c.n; t++) {
            const uint32_t s0 = stage(t);
            if (t + 1 < c.n) {
                if (!mbar_wait(&c.bar[B_FULL0 + ((t + 1) & 1)], ((t + 1) >> 1) & 1, ctl, st, 22)) break;
                if (!mbar_wait(&c.bar[B_PFREE], t & 1, ctl, st, 23)) break;
                tc_fence_after();
                mma1(t + 1);
            }
            if (!mbar_wait(&c.bar[B_SREADY], t & 1, ctl, st, 24)) break;
            if (!mbar_wait(&c.bar[B_WREADY], t & 1, ctl, st, 25)) break;
            tc_fence_after();
            // Delta^T (+)= -S^T W^T
            if (!split) {
                mma_kmn(tm + TM_DL, sa(c, L.sb), 16384, sa(c, L.wb), 16384, 64, 128, true, has_u);
            } else {
                mma_kmn(tm + TM_DL, sa(c, L.sb), 16384, sa(c, L.wb), 16384, 64, 128, true, false);
                mma_kmn(tm + TM_DL, sa(c, L.sb_lo), 16384, sa(c, L.wb), 16384, 64, 128, true, true);
                mma_kmn(tm + TM_DL, sa(c, L.sb), 16384, sa(c, L.wb_lo), 16384, 64, 128, true, true);
            }
            if (fwd) {
                if (t >= 1 && !mbar_wait(&c.bar[B_OFREE], (t - 1) & 1, ctl, st, 26)) break;
                tc_fence_after();
                // O1^T = S^T Q^T
                mma_kk(tm + TM_O1, sa(c, L.sb), 16384, s0 + L.qc0, L.qc1 - L.qc0, 64, 128, false, false);
            }
            mma_commit(&c.bar[B_DLFULL]);
            if (!mbar_wait(&c.bar[B_DLREADY], t & 1, ctl, st, 27)) break;
            tc_fence_after();
            // P_S = (Delta diag Gamma)^T K
            mma_kmn(tm + TM_PS, sa(c, L.dgb), 16384, s0 + L.kc0, L.k_lbo, 128, 64, false, false);
            if (split) mma_kmn(tm + TM_PS, sa(c, L.dgb_lo), 16384, s0 + L.kc0, L.k_lbo, 128, 64, false, true);
            mma_commit(&c.bar[B_PSFULL]);
            if (fwd) {
                if (!mbar_wait(&c.bar[B_MREADY], t & 1, ctl, st, 28)) break;
                tc_fence_after();
                // O2^T = Delta^T mask^T
                mma_kk(tm + TM_O2, sa(c, L.db), 16384, sa(c, L.mask), 8192, 64, 64, false, false);
                mma_commit(&c.bar[B_OFULL]);
                mma_commit(&c.bar[B_MFREE]);
            }
            mma_commit(&c.bar[B_EMPTY0 + (t & 1)]);
            if (t + 1 < c.n) {
                if (!mbar_wait(&c.bar[B_TREADY], (t + 1) & 1, ctl, st, 29)) break;
                tc_fence_after();
                emma(t + 1);
            }
        }
    } while (0);
    // drain every MMA this thread issued
    mma_commit(&c.bar[B_DRAIN]);
    Ctl tmp;
    tmp.abort = 0;
    mbar_wait(&c.bar[B_DRAIN], 0, &tmp, st, 30);
}

// ------------------------------------------------------------------ gates
// Warp 4: beta and g of chunk t, in-chunk cumulative log2 gate G and its
// exponentials into gate slot t % 4 (padded rows: beta = g = 0).
__device__ void compute_gates(const Ctx &c, int t) {
    const int lane = threadIdx.x & 31;
    const int nv = rows_of(c, t);
    Gates gs = gates_of(c.base, c.L, t & 3);
    const int64_t tok = c.f.tok0 + (int64_t)t * C;
    const int H = c.p->H;
    float b0 = 0.f, b1 = 0.f, g0 = 0.f, g1 = 0.f;
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    if (i0 < nv) {
        b0 = __bfloat162float(c.p->beta[(tok + i0) * H + c.h]);
        g0 = c.p->g[(tok + i0) * H + c.h] * kLog2e;
    }
    if (i1 < nv) {
        b1 = __bfloat162float(c.p->beta[(tok + i1) * H + c.h]);
        g1 = c.p->g[(tok + i1) * H + c.h] * kLog2e;
    }
    float x = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    const float G1 = x, G0 = x - g1;
    const float GC = __shfl_sync(0xffffffffu, x, 31);
    gs.G[i0] = G0; gs.G[i1] = G1;
    gs.beta[i0] = b0; gs.beta[i1] = b1;
    gs.gam[i0] = exp2f(G0); gs.gam[i1] = exp2f(G1);
    gs.Gam[i0] = exp2f(GC - G0); gs.Gam[i1] = exp2f(GC - G1);
    if (lane == 0) gs.gC[0] = exp2f(GC);
}

// ------------------------------------------------------------------ solve warpgroup
// In-place inverse of the unit lower-triangular (I + A) held in scr[64][65]
// (strictly lower part = A, the rest 0), by 16x16 blocks: diagonal blocks by
// forward substitution, then block columns right to left,
//   X[ib][jb] = -( sum_{kb = jb+1..ib} X[ib][kb] A[kb][jb] ) X[jb][jb].
// Afterwards scr holds T = (I + A)^-1 with its unit diagonal written out.
__device__ bool solve_inverse(const Ctx &c, uint32_t &wgph) {
    float *S = reinterpret_cast<float *>(c.base + c.L.scr);
    float *Tm = reinterpret_cast<float *>(c.base + c.L.tmp);
    const int t = threadIdx.x - 128;   // 0..127 within the solve warpgroup
    constexpr int LS = 65;
    // diagonal blocks: thread (b, col) for t < 64
    float x[16];
    const int b = t >> 4, col = t & 15;
    if (t < 64) {
        const float *Ab = S + (16 * b) * LS + 16 * b;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < i; k++) s = fmaf(Ab[i * LS + k], x[k], s);
            x[i] = (i < col) ? 0.f : (i == col ? 1.f : -s);
        }
    }
    if (!wg_sync(c, wgph, 40)) return false;
    if (t < 64) {
        float *Ab = S + (16 * b) * LS + 16 * b;
#pragma unroll
        for (int i = 0; i < 16; i++) Ab[i * LS + col] = x[i];
    }
    if (!wg_sync(c, wgph, 41)) return false;
    for (int jb = 2; jb >= 0; jb--) {
        const int r0 = 16 * (jb + 1);           // first row below the diagonal block
        const int R = 64 - r0;                  // rows to fill
        const int cc = t & 15;
        // temp[r][cc] = sum_{k = r0 .. r0 + r} X[r0 + r][k] * A[k][16 jb + cc]
        for (int r = t >> 4; r < R; r += 8) {
            const float *xr = S + (r0 + r) * LS;
            float s = 0.f;
            for (int k = r0; k <= r0 + r; k++) s = fmaf(xr[k], S[k * LS + 16 * jb + cc], s);
            Tm[r * 16 + cc] = s;
        }
        if (!wg_sync(c, wgph, 42)) return false;
        // X[r0 + r][16 jb + cc] = -sum_{m = cc..15} temp[r][m] * X[16 jb + m][16 jb + cc]
        for (int r = t >> 4; r < R; r += 8) {
            float s = 0.f;
            for (int m = cc; m < 16; m++) s = fmaf(Tm[r * 16 + m], S[(16 * jb + m) * LS + 16 * jb + cc], s);
            S[(r0 + r) * LS + 16 * jb + cc] = -s;
        }
        if (!wg_sync(c, wgph, 43)) return false;
    }
    return true;
}

__device__ void run_solve(const Ctx &c) {
    const Lay &L = c.L;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x - 128;
    const bool split = (c.mode == MODE_PRE && c.role == ROLE_M);
    float *S = reinterpret_cast<float *>(c.base + L.scr);
    uint32_t wgph = 0;
    for (int ch = 0; ch < c.n; ch++) {
        const int slot = ch & 3;
        if (w == 4) compute_gates(c, ch);
        if (!wg_sync(c, wgph, 44)) return;
        if (w == 4 && lane == 0) mbar_arrive(&c.bar[B_GATE0 + slot]);
        Gates gs = gates_of(c.base, L, slot);
        // A from K K^T (lanes 0..63 -> warps 4, 5)
        if (!warp_wait(c, B_PFULL, ch & 1, 45)) return;
        tc_fence_after();
        if (w < 6) {
            const int i = 32 * (w - 4) + lane;
            float v[32];
            const float bi = gs.beta[i], Gi = gs.G[i];
#pragma unroll
            for (int half = 0; half < 2; half++) {
                tmem_ld32(c.tmem + ((uint32_t)(32 * (w - 4)) << 16) + TM_P + 32 * half, v);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 32; jj++) {
                    const int j = 32 * half + jj;
                    S[i * 65 + j] = (j < i) ? bi * exp2f(Gi - gs.G[j]) * v[jj] : 0.f;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.bar[B_PFREE]);
        }
        if (!wg_sync(c, wgph, 46)) return;
        if (!solve_inverse(c, wgph)) return;
        // T' = T diag(beta), T'' = T diag(beta gamma) (hi/lo for the split chain), bf16 swizzled
        if (ch >= 1 && !warp_wait(c, B_TFREE, (ch - 1) & 1, 47)) return;
        {
            const int i = t >> 1, hf = t & 1;
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {
                float a[8], bb[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int j = 32 * hf + 8 * q4 + e;
                    const float tij = (j <= i) ? S[i * 65 + j] : 0.f;
                    a[e] = tij * gs.beta[j];
                    bb[e] = a[e] * gs.gam[j];
                }
                const uint32_t off = sw128(i, 4 * hf + q4);
                uint4 hi;
                hi.x = pack_bf16(bb[0], bb[1]); hi.y = pack_bf16(bb[2], bb[3]);
                hi.z = pack_bf16(bb[4], bb[5]); hi.w = pack_bf16(bb[6], bb[7]);
                *reinterpret_cast<uint4 *>(c.base + L.tpp + off) = hi;
                if (split) {
                    const __nv_bfloat162 *hp = reinterpret_cast<const __nv_bfloat162 *>(&hi);
                    float lo[8];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float2 f2 = __bfloat1622float2(hp[e]);
                        lo[2 * e] = bb[2 * e] - f2.x;
                        lo[2 * e + 1] = bb[2 * e + 1] - f2.y;
                    }
                    uint4 lw;
                    lw.x = pack_bf16(lo[0], lo[1]); lw.y = pack_bf16(lo[2], lo[3]);
                    lw.z = pack_bf16(lo[4], lo[5]); lw.w = pack_bf16(lo[6], lo[7]);
                    *reinterpret_cast<uint4 *>(c.base + L.tpp_lo + off) = lw;
                } else {
                    uint4 u;
                    u.x = pack_bf16(a[0], a[1]); u.y = pack_bf16(a[2], a[3]);
                    u.z = pack_bf16(a[4], a[5]); u.w = pack_bf16(a[6], a[7]);
                    *reinterpret_cast<uint4 *>(c.base + L.tp + off) = u;
                }
            }
        }
        fence_async_smem();
        if (!wg_sync(c, wgph, 48)) return;
        if (t == 0) mbar_arrive(&c.bar[B_TREADY]);
        // W epilogue: W^T (lanes = dk) -> bf16 MN-major B tile (hi/lo when split)
        if (!warp_wait(c, B_WFULL, ch & 1, 49)) return;
        tc_fence_after();
        {
            const int dk = 32 * (w - 4) + lane;
#pragma unroll
            for (int half = 0; half < 2; half++) {
                float v[32];
                tmem_ld32(c.tmem + ((uint32_t)(32 * (w - 4)) << 16) + TM_W + 32 * half, v);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {
                    uint4 hi;
                    hi.x = pack_bf16(v[8 * q4 + 0], v[8 * q4 + 1]); hi.y = pack_bf16(v[8 * q4 + 2], v[8 * q4 + 3]);
                    hi.z = pack_bf16(v[8 * q4 + 4], v[8 * q4 + 5]); hi.w = pack_bf16(v[8 * q4 + 6], v[8 * q4 + 7]);
                    const uint32_t off = sw128(dk, 4 * half + q4);
                    *reinterpret_cast<uint4 *>(c.base + L.wb + off) = hi;
                    if (split) {
                        const __nv_bfloat162 *hp = reinterpret_cast<const __nv_bfloat162 *>(&hi);
                        float lo[8];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const float2 f2 = __bfloat1622float2(hp[e]);
                            lo[2 * e] = v[8 * q4 + 2 * e] - f2.x;
                            lo[2 * e + 1] = v[8 * q4 + 2 * e + 1] - f2.y;
                        }
                        uint4 lw;
                        lw.x = pack_bf16(lo[0], lo[1]); lw.y = pack_bf16(lo[2], lo[3]);
                        lw.z = pack_bf16(lo[4], lo[5]); lw.w = pack_bf16(lo[6], lo[7]);
                        *reinterpret_cast<uint4 *>(c.base + L.wb_lo + off) = lw;
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bar[B_WREADY]);
    }
}

// ------------------------------------------------------------------ mask warps (forward)
__device__ void run_mask(const Ctx &c) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = 32 * (w - 2) + lane;   // row of Q K^T (TMEM lane 64 + i)
    for (int ch = 0; ch < c.n; ch++) {
        if (!warp_wait(c, B_GATE0 + (ch & 3), (ch >> 2) & 1, 50)) return;
        Gates gs = gates_of(c.base, c.L, ch & 3);
        if (!warp_wait(c, B_PFULL, ch & 1, 51)) return;
        tc_fence_after();
        float m[64];
        const float Gi = gs.G[i];
#pragma unroll
        for (int half = 0; half < 2; half++) {
            float v[32];
            tmem_ld32(c.tmem + ((uint32_t)(64 + 32 * (w - 2)) << 16) + TM_P + 32 * half, v);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; jj++) {
                const int j = 32 * half + jj;
                m[j] = (j <= i) ? v[jj] * exp2f(Gi - gs.G[j]) : 0.f;
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bar[B_PFREE]);
        if (ch >= 1 && !warp_wait(c, B_MFREE, (ch - 1) & 1, 52)) return;
#pragma unroll
        for (int q = 0; q < 8; q++) {
            uint4 u;
            u.x = pack_bf16(m[8 * q + 0], m[8 * q + 1]); u.y = pack_bf16(m[8 * q + 2], m[8 * q + 3]);
            u.z = pack_bf16(m[8 * q + 4], m[8 * q + 5]); u.w = pack_bf16(m[8 * q + 6], m[8 * q + 7]);
            *reinterpret_cast<uint4 *>(c.base + c.L.mask + sw128(i, q)) = u;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bar[B_MREADY]);
    }
}

// ------------------------------------------------------------------ state warps
// Write 64 fp32 values as one 128-byte bf16 row (8 swizzled chunks) of a
// K-major tile; with `lo_off` also the bf16 residual x - bf16(x).
__device__ __forceinline__ void store_row64(uint8_t *tile, uint8_t *tile_lo, uint32_t row, const float *x) {
#pragma unroll
    for (int q = 0; q < 8; q++) {
        uint4 u;
        u.x = pack_bf16(x[8 * q + 0], x[8 * q + 1]); u.y = pack_bf16(x[8 * q + 2], x[8 * q + 3]);
        u.z = pack_bf16(x[8 * q + 4], x[8 * q + 5]); u.w = pack_bf16(x[8 * q + 6], x[8 * q + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128(row, q)) = u;
        if (tile_lo) {
            const __nv_bfloat162 *hp = reinterpret_cast<const __nv_bfloat162 *>(&u);
            float lo[8];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float2 f2 = __bfloat1622float2(hp[e]);
                lo[2 * e] = x[8 * q + 2 * e] - f2.x;
                lo[2 * e + 1] = x[8 * q + 2 * e + 1] - f2.y;
            }
            uint4 lw;
            lw.x = pack_bf16(lo[0], lo[1]); lw.y = pack_bf16(lo[2], lo[3]);
            lw.z = pack_bf16(lo[4], lo[5]); lw.w = pack_bf16(lo[6], lo[7]);
            *reinterpret_cast<uint4 *>(tile_lo + sw128(row, q)) = lw;
        }
    }
}
// Same for 32 values as chunks [4 half, 4 half + 4) of a row.
__device__ __forceinline__ void store_row32(uint8_t *tile, uint8_t *tile_lo, uint32_t row, int half, const float *x) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint4 u;
        u.x = pack_bf16(x[8 * q + 0], x[8 * q + 1]); u.y = pack_bf16(x[8 * q + 2], x[8 * q + 3]);
        u.z = pack_bf16(x[8 * q + 4], x[8 * q + 5]); u.w = pack_bf16(x[8 * q + 6], x[8 * q + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128(row, 4 * half + q)) = u;
        if (tile_lo) {
            const __nv_bfloat162 *hp = reinterpret_cast<const __nv_bfloat162 *>(&u);
            float lo[8];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float2 f2 = __bfloat1622float2(hp[e]);
                lo[2 * e] = x[8 * q + 2 * e] - f2.x;
                lo[2 * e + 1] = x[8 * q + 2 * e + 1] - f2.y;
            }
            uint4 lw;
            lw.x = pack_bf16(lo[0], lo[1]); lw.y = pack_bf16(lo[2], lo[3]);
            lw.z = pack_bf16(lo[4], lo[5]); lw.w = pack_bf16(lo[6], lo[7]);
            *reinterpret_cast<uint4 *>(tile_lo + sw128(row, 4 * half + q)) = lw;
        }
    }
}

__device__ void run_state(const Ctx &c) {
    const Lay &L = c.L;
    const Params &p = *c.p;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = w & 3, half = (w - 8) >> 2;
    const int row = 32 * q + lane;                       // TMEM lane: value dim (or M column)
    const uint32_t lane_base = c.tmem + ((uint32_t)(32 * q) << 16);
    const bool fwd = c.mode == MODE_FWD, split = (c.mode == MODE_PRE && c.role == ROLE_M);
    const int H = p.H;
    uint8_t *sb = c.base + L.sb + half * 16384, *sb_lo = split ? c.base + L.sb_lo + half * 16384 : nullptr;
    float S[64];
    // initial state: S^T[row][64 half + i]
    {
        const int64_t sidx = ((int64_t)c.f.seg * H + c.h) * D * D;
        for (int i = 0; i < 64; i++) {
            const int dk = 64 * half + i;
            float x = 0.f;
            if (split) x = (dk == row) ? 1.f : 0.f;
            else if (fwd && (c.f.flags & CPDR_FRAG_CONT_PREV)) x = p.S_init[sidx + (int64_t)dk * D + row];
            S[i] = x;
        }
    }
    store_row64(sb, sb_lo, row, S);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.bar[B_SREADY]);
    for (int ch = 0; ch < c.n; ch++) {
        if (!warp_wait(c, B_GATE0 + (ch & 3), (ch >> 2) & 1, 60)) return;
        Gates gs = gates_of(c.base, L, ch & 3);
        // Delta epilogue
        if (!warp_wait(c, B_DLFULL, ch & 1, 61)) return;
        tc_fence_after();
        {
            float v[32], vg[32];
            tmem_ld32(lane_base + TM_DL + 32 * half, v);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; jj++) vg[jj] = v[jj] * gs.Gam[32 * half + jj];
            if (fwd) store_row32(c.base + L.db, nullptr, row, half, v);
            store_row32(c.base + L.dgb, split ? c.base + L.dgb_lo : nullptr, row, half, vg);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bar[B_DLREADY]);
        // state update: S <- gamma^C S + P_S
        if (!warp_wait(c, B_PSFULL, ch & 1, 62)) return;
        tc_fence_after();
        {
            const float gC = gs.gC[0];
#pragma unroll
            for (int piece = 0; piece < 2; piece++) {
                float v[32];
                tmem_ld32(lane_base + TM_PS + 64 * half + 32 * piece, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++) S[32 * piece + i] = fmaf(gC, S[32 * piece + i], v[i]);
            }
        }
        store_row64(sb, sb_lo, row, S);
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bar[B_SREADY]);
        if (fwd) {
            // O = scale (gamma_i O1 + O2)
            if (!warp_wait(c, B_OFULL, ch & 1, 63)) return;
            tc_fence_after();
            float a[32], b[32];
            tmem_ld32(lane_base + TM_O1 + 32 * half, a);
            tmem_ld32(lane_base + TM_O2 + 32 * half, b);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.bar[B_OFREE]);
            const int nv = rows_of(c, ch);
            const int64_t tok = c.f.tok0 + (int64_t)ch * C;
#pragma unroll
            for (int ii = 0; ii < 32; ii++) {
                const int i = 32 * half + ii;
                if (i < nv)
                    p.o[((tok + i) * H + c.h) * D + row] = __float2bfloat16_rn(p.scale * fmaf(gs.gam[i], a[ii], b[ii]));
            }
        }
    }
    // outputs of the chain
    const int64_t sidx = ((int64_t)c.f.seg * H + c.h) * D * D;
    if (fwd) {
        if ((c.f.flags & CPDR_FRAG_ENDS_SEQ) && p.final_state) {
            const int64_t fidx = ((int64_t)c.f.seq * H + c.h) * D * D;
            for (int i = 0; i < 64; i++) p.final_state[fidx + (int64_t)(64 * half + i) * D + row] = S[i];
        }
    } else {
        float *dst = split ? p.M : p.S_ext;
        for (int i = 0; i < 64; i++) dst[sidx + (int64_t)(64 * half + i) * D + row] = S[i];
    }
}

// ------------------------------------------------------------------ kernel
template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
tc_chain_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int role = MODE == MODE_PRE ? (int)(blockIdx.x & 1) : ROLE_S;
    const int item = MODE == MODE_PRE ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    Ctx c;
    c.base = base;
    c.L = make_lay(MODE, role);
    c.bar = reinterpret_cast<uint64_t *>(base + c.L.bars);
    c.ctl = reinterpret_cast<Ctl *>(base + c.L.bars + NBARS * 8);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + c.L.bars + NBARS * 8 + 16);
    c.mode = MODE;
    c.role = role;
    c.f = p.frags[p.items[item]];
    c.h = blockIdx.y;
    c.n = (c.f.len + C - 1) / C;
    c.nlast = c.f.len - (c.n - 1) * C;
    c.p = &p;
    const int w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        const int fwd = MODE == MODE_FWD;
        const uint32_t cnt[NBARS] = {1, 1, 1, 1, 1, (uint32_t)(fwd ? 4 : 2), 1, 1, 2, 1,
                                     1, 4, 1, 8, 1, 8, 1, 8,
                                     1, 1, 1, 1, 4, 1};
        for (int i = 0; i < NBARS; i++) mbar_init(&c.bar[i], cnt[i]);
        c.ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 0 && (threadIdx.x & 31) == 0) {
        tma_prefetch_desc(&tk);
        if (MODE == MODE_FWD) tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tv);
    }
    if (w == 1) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tmem_slot;
    if (w == 0) run_producer(c, &tq, &tk, &tv);
    else if (w == 1) run_mma(c);
    else if (w < 4) { if (MODE == MODE_FWD) run_mask(c); }
    else if (w < 8) run_solve(c);
    else run_state(c);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == 1) tmem_dealloc(c.tmem, TM_COLS);
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

size_t smem_for(int mode) {
    size_t a = make_lay(mode, ROLE_S).total, b = make_lay(mode, ROLE_M).total;
    return (mode == MODE_FWD ? a : (a > b ? a : b)) + 1024;
}

}  // namespace

bool tc_supported(const Plan &p) {
    return p.in_dtype == CPDR_DTYPE_BF16 && p.dk == 128 && p.dv == 128 && p.gate_kind == CPDR_GATE_SCALAR;
}

int launch_tc_pre(const cpdr_ctx *c, const void *k, const void *v, const void *beta, const float *g, float *S_ext,
                  float *M, void *stream) {
    const auto &p = c->plan;
    if (p.pre_items.empty()) return 0;
    CUtensorMap tk, tv;
    const int64_t tokens = (int64_t)p.B * p.T;
    if (!make_tmap(&tk, k, tokens, p.H) || !make_tmap(&tv, v, tokens, p.H)) return (int)cudaErrorInvalidValue;
    Params prm{};
    prm.frags = c->dev.frags;
    prm.items = c->dev.pre_items;
    prm.beta = (const __nv_bfloat16 *)beta;
    prm.g = g;
    prm.S_ext = S_ext;
    prm.M = M;
    prm.status = c->dev.status;
    prm.H = p.H;
    prm.scale = p.scale;
    const size_t sm = smem_for(MODE_PRE);
    cudaError_t e = cudaFuncSetAttribute(tc_chain_kernel<MODE_PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((unsigned)(2 * p.pre_items.size()), (unsigned)p.H);
    tc_chain_kernel<MODE_PRE><<<grid, NTHREADS, sm, (cudaStream_t)stream>>>(tk, tk, tv, prm);
    return (int)cudaGetLastError();
}

int launch_tc_fwd(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta, const float *g,
                  const float *S_init, void *o, float *final_state, void *stream) {
    const auto &p = c->plan;
    if (p.frags.empty()) return 0;
    CUtensorMap tq, tk, tv;
    const int64_t tokens = (int64_t)p.B * p.T;
    if (!make_tmap(&tq, q, tokens, p.H) || !make_tmap(&tk, k, tokens, p.H) || !make_tmap(&tv, v, tokens, p.H))
        return (int)cudaErrorInvalidValue;
    Params prm{};
    prm.frags = c->dev.frags;
    prm.items = c->dev.fwd_order;
    prm.beta = (const __nv_bfloat16 *)beta;
    prm.g = g;
    prm.S_init = S_init;
    prm.o = (__nv_bfloat16 *)o;
    prm.final_state = final_state;
    prm.status = c->dev.status;
    prm.H = p.H;
    prm.scale = p.scale;
    const size_t sm = smem_for(MODE_FWD);
    cudaError_t e = cudaFuncSetAttribute(tc_chain_kernel<MODE_FWD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((unsigned)p.frags.size(), (unsigned)p.H);
    tc_chain_kernel<MODE_FWD><<<grid, NTHREADS, sm, (cudaStream_t)stream>>>(tq, tk, tv, prm);
    return (int)cudaGetLastError();
}

}  // namespace cpdr
