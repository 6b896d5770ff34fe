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
// registers, 64 values per thread).  Roles and shared-memory layouts are
// compile-time and every role function is inlined, so per-CTA state stays in
// registers.  Every mbarrier wait is bounded: on expiry the kernel records a
// status code, raises an abort flag that makes every other wait fall
// through, drains its MMAs and loads, frees TMEM and returns.  The solve
// warpgroup synchronises with a hardware named barrier; its mbarrier waits
// are taken by one warp and the verdict is broadcast across that barrier, so
// an abort can never strand a warp inside it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"

// Optional event trace (compile with -DCPDR_TRACE): CTA (0, 0) of each
// launch records %globaltimer stamps per role, chunk and event.
#ifdef CPDR_TRACE
__device__ unsigned long long g_cpdr_trace[3][8][64][16];
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define TR(role, chunk, ev)                                                                \
    do {                                                                                   \
        if (blockIdx.x == 0 && blockIdx.y == 0 && (threadIdx.x & 31) == 0 && (chunk) < 64) \
            g_cpdr_trace[MODE * (1 + ROLE)][role][chunk][ev] = gtimer();                                \
    } while (0)
#else
#define TR(role, chunk, ev) \
    do {                    \
    } while (0)
#endif

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
    B_GATE0, B_GATE1, B_GATE2, B_GATE3, B_DRAIN, NBARS
};
constexpr int kSolveBar = 1;   // named barrier id of the solve warpgroup

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
    uint32_t tp, tpp, tpp_lo, mask, wb, wb_lo, sb, sb_lo, db, dgb, dgb_lo, scr, tmp, gates, graw, bars, ctl, verdict,
        tslot, total;
};

__host__ __device__ constexpr Lay make_lay(int mode, int role) {
    Lay L{};
    if (mode == MODE_FWD) {
        L.stage_bytes = 49152; L.kc0 = 0; L.qc0 = 8192; L.kc1 = 16384; L.qc1 = 24576; L.vc0 = 32768; L.vc1 = 40960;
        L.k_lbo = 16384; L.v_lbo = 8192; L.tx_bytes = 49152;
    } else if (role == ROLE_S) {
        L.stage_bytes = 32768; L.kc0 = 0; L.vc0 = 8192; L.kc1 = 16384; L.vc1 = 24576; L.qc0 = 0; L.qc1 = 0;
        L.k_lbo = 16384; L.v_lbo = 16384; L.tx_bytes = 32768;
    } else {
        L.stage_bytes = 16384; L.kc0 = 0; L.kc1 = 8192; L.qc0 = 0; L.qc1 = 0; L.vc0 = 0; L.vc1 = 0;
        L.k_lbo = 8192; L.v_lbo = 0; L.tx_bytes = 16384;
    }
    uint32_t o = 2 * L.stage_bytes;
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
    L.scr = o; o += 64 * 68 * 4;              // solve scratch, fp32 [64][68] (16-byte rows)
    L.tmp = o; o += 48 * 16 * 4;              // solve temporary
    L.gates = o; o += 4 * (4 * 64 + 4) * 4;   // 4 slots: G, beta, gamma, Gamma, gamma^C
    L.graw = o; o += 2 * 128 * 4;             // per stage: raw beta[64], log2 gate[64]
    o = (o + 15) & ~15u;
    L.bars = o; o += NBARS * 8;
    L.ctl = o; o += 16;
    L.verdict = o; o += 16;
    L.tslot = o; o += 16;
    L.total = o;
    return L;
}

// Per-CTA runtime state (registers once every role function is inlined).
struct Run {
    uint8_t *base;
    uint64_t *bar;
    Ctl *ctl;
    uint32_t tmem;
    int n, nlast, h;
    int64_t tok0;
    int seg, seq, flags;
    const Params *p;
};

// gate slot arrays
struct Gates {
    float *G, *beta, *gam, *Gam, *gC;
};
template <int MODE, int ROLE>
__device__ __forceinline__ Gates gates_of(const Run &r, int slot) {
    constexpr Lay L = make_lay(MODE, ROLE);
    float *q = reinterpret_cast<float *>(r.base + L.gates) + slot * (4 * 64 + 4);
    return Gates{q, q + 64, q + 128, q + 192, q + 256};
}

__device__ __forceinline__ int rows_of(const Run &r, int chunk) { return chunk == r.n - 1 ? r.nlast : C; }

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast, then
// every lane performs its own (now immediate) acquire.
__device__ __forceinline__ bool warp_wait(const Run &r, int b, uint32_t parity, int site) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(&r.bar[b], parity, r.ctl, r.p->status, site) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(&r.bar[b], parity);
    return ok != 0;
}

// Solve-warpgroup wait: warp 4 waits (bounded), writes the verdict, and the
// named barrier publishes it to warps 5..7.  Two alternating verdict slots.
__device__ __forceinline__ bool group_wait(const Run &r, volatile int *verdict, int &vslot, int b, uint32_t parity,
                                           int site) {
    volatile int *v = verdict + (vslot & 1);
    vslot++;
    if ((threadIdx.x >> 5) == 4) {
        const bool ok = warp_wait(r, b, parity, site);
        if ((threadIdx.x & 31) == 0) *v = ok ? 1 : 0;
    }
    named_bar(kSolveBar, 128);
    const int ok = *v;
    if (ok) mbar_try_wait(&r.bar[b], parity);
    return ok != 0;
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

// ------------------------------------------------------------------ producer
template <int MODE, int ROLE>
__device__ __forceinline__ void run_producer(const Run &r, const CUtensorMap *tq, const CUtensorMap *tk,
                                             const CUtensorMap *tv) {
    constexpr Lay L = make_lay(MODE, ROLE);
    const int lane = threadIdx.x & 31;
    const int H = r.p->H;
    int issued[2] = {-1, -1};
    for (int t = 0; t < r.n; t++) {
        const int s = t & 1;
        int ok = 1;
        if (lane == 0 && t >= 2) ok = mbar_wait(&r.bar[B_EMPTY0 + s], ((t >> 1) - 1) & 1, r.ctl, r.p->status, 10);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        TR(0, t, 0);
        uint64_t *fb = &r.bar[B_FULL0 + s];
        const int tok = (int)(r.tok0 + (int64_t)t * C);
        if (lane == 0) {
            uint8_t *st = r.base + s * L.stage_bytes;
            mbar_arrive_expect_tx(fb, L.tx_bytes);
            tma_load_3d(st + L.kc0, tk, fb, 0, r.h, tok);
            tma_load_3d(st + L.kc1, tk, fb, 64, r.h, tok);
            if (MODE == MODE_FWD) {
                tma_load_3d(st + L.qc0, tq, fb, 0, r.h, tok);
                tma_load_3d(st + L.qc1, tq, fb, 64, r.h, tok);
            }
            if (MODE == MODE_FWD || ROLE == ROLE_S) {
                tma_load_3d(st + L.vc0, tv, fb, 0, r.h, tok);
                tma_load_3d(st + L.vc1, tv, fb, 64, r.h, tok);
            }
        }
        // beta and the log2 gate of the chunk's rows (padded rows: 0), second arrival on FULL
        {
            const int nv = rows_of(r, t);
            float *raw = reinterpret_cast<float *>(r.base + L.graw) + s * 128;
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int i = lane + 32 * e;
                float b = 0.f, gg = 0.f;
                if (i < nv) {
                    b = __bfloat162float(r.p->beta[((int64_t)tok + i) * H + r.h]);
                    gg = r.p->g[((int64_t)tok + i) * H + r.h] * kLog2e;
                }
                raw[i] = b;
                raw[64 + i] = gg;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(fb);
        }
        issued[s] = t;
    }
    // drain: every issued load must have landed before the CTA exits
    if (lane == 0) {
        Ctl local;
        local.abort = 0;
        for (int s = 0; s < 2; s++)
            if (issued[s] >= 0) mbar_wait(&r.bar[B_FULL0 + s], (issued[s] >> 1) & 1, &local, r.p->status, 11);
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

template <int MODE, int ROLE>
__device__ __forceinline__ void run_mma(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool FWD = MODE == MODE_FWD, SPLIT = (MODE == MODE_PRE && ROLE == ROLE_M);
    constexpr bool HAS_U = FWD || ROLE == ROLE_S;
    if ((threadIdx.x & 31) != 0) return;
    const uint32_t tm = r.tmem;
    int32_t *st = r.p->status;
    Ctl *ctl = r.ctl;
    const uint32_t b0 = smem_u32(r.base);
    // per-stage operand descriptors (stage 1 = stage 0 + stage_bytes >> 4)
    const uint64_t d_stack0 = kdesc(b0 + L.kc0), d_kmn0 = mndesc(b0 + L.kc0, L.k_lbo);
    const uint64_t d_vmn0 = mndesc(b0 + L.vc0, L.v_lbo), d_q0 = kdesc(b0 + L.qc0);
    auto stg = [&](uint64_t d, int t) { return d + (uint64_t)((t & 1) * (L.stage_bytes >> 4)); };
    const uint64_t d_tp = kdesc(b0 + L.tp), d_tpp = kdesc(b0 + L.tpp), d_tpplo = kdesc(b0 + L.tpp_lo);
    const uint64_t d_sb = kdesc(b0 + L.sb), d_sblo = kdesc(b0 + L.sb_lo);
    const uint64_t d_wb = mndesc(b0 + L.wb, 16384), d_wblo = mndesc(b0 + L.wb_lo, 16384);
    const uint64_t d_dgb = kdesc(b0 + L.dgb), d_dgblo = kdesc(b0 + L.dgb_lo), d_db = kdesc(b0 + L.db);
    const uint64_t d_mask = kdesc(b0 + L.mask);
    constexpr uint32_t KATOM = L.kc1 - L.kc0, QATOM = L.qc1 - L.qc0;

    auto mma1 = [&](int t) {   // P = [K; Q] K^T  (rows 64..127 of the A tile: Q, V or unused)
        mma_kk<64, 128, false>(tm + TM_P, stg(d_stack0, t), KATOM, stg(d_stack0, t), KATOM, false);
        mma_commit(&r.bar[B_PFULL]);
    };
    auto emma = [&](int t) {   // W^T = K^T T''^T (hi + lo when split), U^T = V^T T'^T
        mma_mnk<64, 64>(tm + TM_W, stg(d_kmn0, t), d_tpp, 8192, false);
        if (SPLIT) mma_mnk<64, 64>(tm + TM_W, stg(d_kmn0, t), d_tpplo, 8192, true);
        mma_commit(&r.bar[B_WFULL]);
        if (HAS_U) mma_mnk<64, 64>(tm + TM_DL, stg(d_vmn0, t), d_tp, 8192, false);
        mma_commit(&r.bar[B_TFREE]);
    };
    do {
        if (!mbar_wait(&r.bar[B_FULL0], 0, ctl, st, 20)) break;
        tc_fence_after();
        mma1(0);
        if (!mbar_wait(&r.bar[B_TREADY], 0, ctl, st, 21)) break;
        tc_fence_after();
        emma(0);
        for (int t = 0; t < r.n; t++) {
            const int s = t & 1;
            if (t + 1 < r.n) {
                if (!mbar_wait(&r.bar[B_FULL0 + ((t + 1) & 1)], ((t + 1) >> 1) & 1, ctl, st, 22)) break;
                if (!mbar_wait(&r.bar[B_PFREE], t & 1, ctl, st, 23)) break;
                tc_fence_after();
                mma1(t + 1);
            }
            TR(1, t, 0);
            if (!mbar_wait(&r.bar[B_SREADY], t & 1, ctl, st, 24)) break;
            TR(1, t, 1);
            if (!mbar_wait(&r.bar[B_WREADY], t & 1, ctl, st, 25)) break;
            TR(1, t, 2);
            tc_fence_after();
            // Delta^T (+)= -S^T W^T
            if (!SPLIT) {
                mma_kmn<64, 128, true>(tm + TM_DL, d_sb, 16384, d_wb, HAS_U);
            } else {
                mma_kmn<64, 128, true>(tm + TM_DL, d_sb, 16384, d_wb, false);
                mma_kmn<64, 128, true>(tm + TM_DL, d_sblo, 16384, d_wb, true);
                mma_kmn<64, 128, true>(tm + TM_DL, d_sb, 16384, d_wblo, true);
            }
            if (FWD) {
                if (t >= 1 && !mbar_wait(&r.bar[B_OFREE], (t - 1) & 1, ctl, st, 26)) break;
                tc_fence_after();
                mma_kk<64, 128, false>(tm + TM_O1, d_sb, 16384, stg(d_q0, t), QATOM, false);   // O1^T = S^T Q^T
            }
            mma_commit(&r.bar[B_DLFULL]);
            TR(1, t, 3);
            if (!mbar_wait(&r.bar[B_DLREADY], t & 1, ctl, st, 27)) break;
            TR(1, t, 4);
            tc_fence_after();
            // P_S = (Delta diag Gamma)^T K
            mma_kmn<128, 64, false>(tm + TM_PS, d_dgb, 16384, stg(d_kmn0, t), false);
            if (SPLIT) mma_kmn<128, 64, false>(tm + TM_PS, d_dgblo, 16384, stg(d_kmn0, t), true);
            mma_commit(&r.bar[B_PSFULL]);
            if (FWD) {
                if (!mbar_wait(&r.bar[B_MREADY], t & 1, ctl, st, 28)) break;
                tc_fence_after();
                mma_kk<64, 64, false>(tm + TM_O2, d_db, 16384, d_mask, 8192, false);   // O2^T = Delta^T mask^T
                mma_commit(&r.bar[B_OFULL]);
                mma_commit(&r.bar[B_MFREE]);
            }
            mma_commit(&r.bar[B_EMPTY0 + s]);
            TR(1, t, 5);
            if (t + 1 < r.n) {
                if (!mbar_wait(&r.bar[B_TREADY], (t + 1) & 1, ctl, st, 29)) break;
                TR(1, t, 6);
                tc_fence_after();
                emma(t + 1);
            }
        }
    } while (0);
    // drain every MMA this thread issued
    mma_commit(&r.bar[B_DRAIN]);
    Ctl local;
    local.abort = 0;
    mbar_wait(&r.bar[B_DRAIN], 0, &local, st, 30);
}

// ------------------------------------------------------------------ gates
// Warp 4: in-chunk cumulative log2 gate G of chunk t and its exponentials,
// from the raw beta / log2 gate the producer warp staged with the chunk,
// into gate slot t % 4.  Padded rows carry beta = g = 0.
__device__ __forceinline__ void write_gates(const Gates &gs, const float *raw) {
    const int lane = threadIdx.x & 31;
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    const float2 bb = *reinterpret_cast<const float2 *>(raw + i0);
    const float2 gg = *reinterpret_cast<const float2 *>(raw + 64 + i0);
    float x = gg.x + gg.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    const float G1 = x, G0 = x - gg.y;
    const float GC = __shfl_sync(0xffffffffu, x, 31);
    gs.G[i0] = G0; gs.G[i1] = G1;
    gs.beta[i0] = bb.x; gs.beta[i1] = bb.y;
    gs.gam[i0] = exp2f(G0); gs.gam[i1] = exp2f(G1);
    gs.Gam[i0] = exp2f(GC - G0); gs.Gam[i1] = exp2f(GC - G1);
    if (lane == 0) gs.gC[0] = exp2f(GC);
}

// ------------------------------------------------------------------ solve warpgroup
// In-place inverse of the unit lower-triangular (I + A) held in scr[64][68]
// (strictly lower part = A, the rest 0), by 16x16 blocks: diagonal blocks by
// forward substitution, then block columns right to left,
//   X[ib][jb] = -( sum_{kb = jb+1..ib} X[ib][kb] A[kb][jb] ) X[jb][jb].
// Afterwards scr holds T = (I + A)^-1 with its unit diagonal written out.

// One block column JB (rows below the diagonal block):
//   temp[r][cc] = sum_k X[r0 + r][k] A[k][16 JB + cc]     (X lower, upper part 0)
//   X[r0 + r][16 JB + cc] = -sum_m temp[r][m] X[16 JB + m][16 JB + cc]
// Each thread owns column cc and rows t/16 + 8 m, all m interleaved for ILP.
template <int JB>
__device__ __forceinline__ void solve_block_column(float *S, float *Tm, int t) {
    constexpr int LS = 68, r0 = 16 * (JB + 1), R = 64 - r0, NM = R / 8;
    const int cc = t & 15, rb = t >> 4;
    float acc[NM];
#pragma unroll
    for (int m = 0; m < NM; m++) acc[m] = 0.f;
#pragma unroll 2
    for (int k = r0; k < 64; k += 4) {
        const float a0 = S[k * LS + 16 * JB + cc], a1 = S[(k + 1) * LS + 16 * JB + cc];
        const float a2 = S[(k + 2) * LS + 16 * JB + cc], a3 = S[(k + 3) * LS + 16 * JB + cc];
#pragma unroll
        for (int m = 0; m < NM; m++) {
            const float4 x = *reinterpret_cast<const float4 *>(S + (r0 + rb + 8 * m) * LS + k);
            acc[m] = fmaf(x.x, a0, acc[m]);
            acc[m] = fmaf(x.y, a1, acc[m]);
            acc[m] = fmaf(x.z, a2, acc[m]);
            acc[m] = fmaf(x.w, a3, acc[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < NM; m++) Tm[(rb + 8 * m) * 16 + cc] = acc[m];
    named_bar(kSolveBar, 128);
#pragma unroll
    for (int m = 0; m < NM; m++) acc[m] = 0.f;
#pragma unroll 4
    for (int mm = 0; mm < 16; mm++) {
        const float x = S[(16 * JB + mm) * LS + 16 * JB + cc];
#pragma unroll
        for (int m = 0; m < NM; m++) acc[m] = fmaf(Tm[(rb + 8 * m) * 16 + mm], x, acc[m]);
    }
#pragma unroll
    for (int m = 0; m < NM; m++) S[(r0 + rb + 8 * m) * LS + 16 * JB + cc] = -acc[m];
    named_bar(kSolveBar, 128);
}

__device__ __forceinline__ void solve_inverse(float *S, float *Tm, int t) {
    constexpr int LS = 68;
    float x[16];
    const int b = t >> 4, col = t & 15;
    if (t < 64) {   // diagonal block b, column col
        const float *Ab = S + (16 * b) * LS + 16 * b;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < i; k++) s = fmaf(Ab[i * LS + k], x[k], s);
            x[i] = (i < col) ? 0.f : (i == col ? 1.f : -s);
        }
    }
    named_bar(kSolveBar, 128);
    if (t < 64) {
        float *Ab = S + (16 * b) * LS + 16 * b;
#pragma unroll
        for (int i = 0; i < 16; i++) Ab[i * LS + col] = x[i];
    }
    named_bar(kSolveBar, 128);
    solve_block_column<2>(S, Tm, t);
    solve_block_column<1>(S, Tm, t);
    solve_block_column<0>(S, Tm, t);
}

template <int MODE, int ROLE>
__device__ __forceinline__ void run_solve(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool SPLIT = (MODE == MODE_PRE && ROLE == ROLE_M);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x - 128;
    float *S = reinterpret_cast<float *>(r.base + L.scr);
    float *Tm = reinterpret_cast<float *>(r.base + L.tmp);
    volatile int *verdict = reinterpret_cast<volatile int *>(r.base + L.verdict);
    int vslot = 0;
    for (int ch = 0; ch < r.n; ch++) {
        const int slot = ch & 3;
        const Gates gs = gates_of<MODE, ROLE>(r, slot);
        if (w == 4) {
            TR(2, ch, 0);
            if (!warp_wait(r, B_FULL0 + (ch & 1), (ch >> 1) & 1, 44)) return;
            write_gates(gs, reinterpret_cast<const float *>(r.base + L.graw) + (ch & 1) * 128);
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.bar[B_GATE0 + slot]);
            TR(2, ch, 1);
        }
        if (!group_wait(r, verdict, vslot, B_PFULL, ch & 1, 45)) return;
        TR(2, ch, 2);
        tc_fence_after();
        // A from K K^T (TMEM lanes 0..63 -> warps 4, 5)
        if (w < 6) {
            const int i = 32 * (w - 4) + lane;
            const float bi = gs.beta[i], Gi = gs.G[i];
#pragma unroll 1
            for (int half = 0; half < 2; half++) {
                float v[32];
                tmem_ld32(r.tmem + ((uint32_t)(32 * (w - 4)) << 16) + TM_P + 32 * half, v);
                float Gj[32];
#pragma unroll
                for (int q4 = 0; q4 < 8; q4++) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(gs.G + 32 * half + 4 * q4);
                    Gj[4 * q4] = g4.x; Gj[4 * q4 + 1] = g4.y; Gj[4 * q4 + 2] = g4.z; Gj[4 * q4 + 3] = g4.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 8; q4++) {
                    float e[4];
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const int jj = 4 * q4 + u, j = 32 * half + jj;
                        e[u] = (j < i) ? bi * exp2f(Gi - Gj[jj]) * v[jj] : 0.f;
                    }
                    *reinterpret_cast<float4 *>(S + i * 68 + 32 * half + 4 * q4) = make_float4(e[0], e[1], e[2], e[3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.bar[B_PFREE]);
        }
        named_bar(kSolveBar, 128);
        TR(2, ch, 3);
        solve_inverse(S, Tm, t);
        TR(2, ch, 4);
        // T' = T diag(beta), T'' = T diag(beta gamma) (hi/lo when split), bf16 swizzled
        if (ch >= 1 && !group_wait(r, verdict, vslot, B_TFREE, (ch - 1) & 1, 47)) return;
        {
            const int i = t >> 1, hf = t & 1;
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {
                float a[8], bb[8];
#pragma unroll
                for (int e4 = 0; e4 < 2; e4++) {
                    const int j0 = 32 * hf + 8 * q4 + 4 * e4;
                    const float4 t4 = *reinterpret_cast<const float4 *>(S + i * 68 + j0);
                    const float4 b4 = *reinterpret_cast<const float4 *>(gs.beta + j0);
                    const float4 g4 = *reinterpret_cast<const float4 *>(gs.gam + j0);
                    const float tv[4] = {t4.x, t4.y, t4.z, t4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
                    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const float tij = (j0 + u <= i) ? tv[u] : 0.f;
                        a[4 * e4 + u] = tij * bv[u];
                        bb[4 * e4 + u] = a[4 * e4 + u] * gv[u];
                    }
                }
                const uint32_t off = sw128(i, 4 * hf + q4);
                const uint4 hi = pack8(bb);
                *reinterpret_cast<uint4 *>(r.base + L.tpp + off) = hi;
                if (SPLIT) *reinterpret_cast<uint4 *>(r.base + L.tpp_lo + off) = pack8_residual(bb, hi);
                else *reinterpret_cast<uint4 *>(r.base + L.tp + off) = pack8(a);
            }
        }
        fence_async_smem();
        named_bar(kSolveBar, 128);
        if (t == 0) mbar_arrive(&r.bar[B_TREADY]);
        TR(2, ch, 5);
        // W epilogue: W^T (lanes = dk) -> bf16 MN-major B tile (hi/lo when split)
        if (!group_wait(r, verdict, vslot, B_WFULL, ch & 1, 49)) return;
        TR(2, ch, 6);
        tc_fence_after();
        {
            const int dk = 32 * (w - 4) + lane;
#pragma unroll 1
            for (int half = 0; half < 2; half++) {
                float v[32];
                tmem_ld32(r.tmem + ((uint32_t)(32 * (w - 4)) << 16) + TM_W + 32 * half, v);
                tmem_ld_wait();
                store_row<4>(r.base + L.wb, SPLIT ? r.base + L.wb_lo : nullptr, dk, 4 * half, v);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_WREADY]);
        TR(2, ch, 7);
    }
}

// ------------------------------------------------------------------ mask warps (forward)
template <int MODE, int ROLE>
__device__ __forceinline__ void run_mask(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = 32 * (w - 2) + lane;   // row of Q K^T (TMEM lane 64 + i)
    for (int ch = 0; ch < r.n; ch++) {
        if (!warp_wait(r, B_GATE0 + (ch & 3), (ch >> 2) & 1, 50)) return;
        const Gates gs = gates_of<MODE, ROLE>(r, ch & 3);
        if (w == 2) TR(4, ch, 0);
        if (!warp_wait(r, B_PFULL, ch & 1, 51)) return;
        if (w == 2) TR(4, ch, 1);
        tc_fence_after();
        const float Gi = gs.G[i];
        float m[64];
#pragma unroll
        for (int half = 0; half < 2; half++) {
            float v[32];
            tmem_ld32(r.tmem + ((uint32_t)(64 + 32 * (w - 2)) << 16) + TM_P + 32 * half, v);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 8; q4++) {
                const float4 g4 = *reinterpret_cast<const float4 *>(gs.G + 32 * half + 4 * q4);
                const float gj[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const int jj = 4 * q4 + u, j = 32 * half + jj;
                    m[j] = (j <= i) ? v[jj] * exp2f(Gi - gj[u]) : 0.f;
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

// ------------------------------------------------------------------ state warps
template <int MODE, int ROLE>
__device__ __forceinline__ void run_state(const Run &r) {
    constexpr Lay L = make_lay(MODE, ROLE);
    constexpr bool FWD = MODE == MODE_FWD, SPLIT = (MODE == MODE_PRE && ROLE == ROLE_M);
    const Params &p = *r.p;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = w & 3, half = (w - 8) >> 2;
    const int row = 32 * q + lane;                       // TMEM lane: value dim (or M column)
    const uint32_t lane_base = r.tmem + ((uint32_t)(32 * q) << 16);
    const int H = p.H;
    uint8_t *sb = r.base + L.sb + half * 16384;
    uint8_t *sb_lo = SPLIT ? r.base + L.sb_lo + half * 16384 : nullptr;
    float S[64];
    const int64_t sidx = ((int64_t)r.seg * H + r.h) * D * D;
    // initial state: S^T[row][64 half + i]
#pragma unroll
    for (int i = 0; i < 64; i++) {
        const int dk = 64 * half + i;
        float x = 0.f;
        if (SPLIT) x = (dk == row) ? 1.f : 0.f;
        else if (FWD && (r.flags & CPDR_FRAG_CONT_PREV)) x = p.S_init[sidx + (int64_t)dk * D + row];
        S[i] = x;
    }
    store_row<8>(sb, sb_lo, row, 0, S);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&r.bar[B_SREADY]);
    for (int ch = 0; ch < r.n; ch++) {
        if (!warp_wait(r, B_GATE0 + (ch & 3), (ch >> 2) & 1, 60)) return;
        const Gates gs = gates_of<MODE, ROLE>(r, ch & 3);
        // Delta epilogue
        if (w == 8) TR(3, ch, 0);
        if (!warp_wait(r, B_DLFULL, ch & 1, 61)) return;
        if (w == 8) TR(3, ch, 1);
        tc_fence_after();
        {
            float v[32];
            tmem_ld32(lane_base + TM_DL + 32 * half, v);
            tmem_ld_wait();
            if (FWD) store_row<4>(r.base + L.db, nullptr, row, 4 * half, v);
#pragma unroll
            for (int jj = 0; jj < 32; jj++) v[jj] *= gs.Gam[32 * half + jj];
            store_row<4>(r.base + L.dgb, SPLIT ? r.base + L.dgb_lo : nullptr, row, 4 * half, v);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_DLREADY]);
        if (w == 8) TR(3, ch, 2);
        // state update: S <- gamma^C S + P_S
        if (!warp_wait(r, B_PSFULL, ch & 1, 62)) return;
        if (w == 8) TR(3, ch, 3);
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
        store_row<8>(sb, sb_lo, row, 0, S);
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.bar[B_SREADY]);
        if (w == 8) TR(3, ch, 4);
        if (FWD) {
            // O = scale (gamma_i O1 + O2)
            if (!warp_wait(r, B_OFULL, ch & 1, 63)) return;
            tc_fence_after();
            const int nv = rows_of(r, ch) - 32 * half;   // valid rows of this thread's half
            const int64_t ostride = (int64_t)H * D;
            __nv_bfloat16 *op = p.o + ((r.tok0 + (int64_t)ch * C + 32 * half) * H + r.h) * D + row;
            const float sc = p.scale;
            const float *gam = gs.gam + 32 * half;
#pragma unroll
            for (int piece = 0; piece < 2; piece++) {
                float a[16], b[16];
                tmem_ld16(lane_base + TM_O1 + 32 * half + 16 * piece, a);
                tmem_ld16(lane_base + TM_O2 + 32 * half + 16 * piece, b);
                tmem_ld_wait();
                if (piece == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&r.bar[B_OFREE]);
                }
#pragma unroll
                for (int ii = 0; ii < 16; ii++) {
                    const int i = 16 * piece + ii;
                    if (i < nv) op[i * ostride] = __float2bfloat16_rn(sc * fmaf(gam[i], a[ii], b[ii]));
                }
            }
            if (w == 8) TR(3, ch, 5);
        }
    }
    // outputs of the chain
    if (FWD) {
        if ((r.flags & CPDR_FRAG_ENDS_SEQ) && p.final_state) {
            const int64_t fidx = ((int64_t)r.seq * H + r.h) * D * D;
#pragma unroll
            for (int i = 0; i < 64; i++) p.final_state[fidx + (int64_t)(64 * half + i) * D + row] = S[i];
        }
    } else {
        float *dst = SPLIT ? p.M : p.S_ext;
#pragma unroll
        for (int i = 0; i < 64; i++) dst[sidx + (int64_t)(64 * half + i) * D + row] = S[i];
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
    const cpdr_fragment f = p.frags[p.items[item]];
    r.tok0 = f.tok0;
    r.seg = f.seg;
    r.seq = f.seq;
    r.flags = f.flags;
    r.h = blockIdx.y;
    r.n = (f.len + C - 1) / C;
    r.nlast = f.len - (r.n - 1) * C;
    r.p = &p;
    if (threadIdx.x == 0) {
        const uint32_t cnt[NBARS] = {2, 2, 1, 1, 1, (uint32_t)(MODE == MODE_FWD ? 4 : 2), 1, 1, 2, 1,
                                     1, 4, 1, 8, 1, 8, 1, 8,
                                     1, 1, 1, 1, 1};
        for (int i = 0; i < NBARS; i++) mbar_init(&r.bar[i], cnt[i]);
        r.ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 0 && (threadIdx.x & 31) == 0) {
        tma_prefetch_desc(tk);
        if (MODE == MODE_FWD) tma_prefetch_desc(tq);
        if (MODE == MODE_FWD || ROLE == ROLE_S) tma_prefetch_desc(tv);
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
    else if (w < 4) { if (MODE == MODE_FWD) run_mask<MODE, ROLE>(r); }
    else if (w < 8) run_solve<MODE, ROLE>(r);
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

size_t smem_for(int mode, int role) { return make_lay(mode, role).total + 1024; }

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
    // the S chains and the transfer-matrix chains, one kernel each
    int rc = launch_chain<MODE_PRE, ROLE_S>(tk, tk, tv, prm, (unsigned)p.pre_items.size(), (unsigned)p.H,
                                            (cudaStream_t)stream);
    if (rc) return rc;
    return launch_chain<MODE_PRE, ROLE_M>(tk, tk, tv, prm, (unsigned)p.pre_items.size(), (unsigned)p.H,
                                          (cudaStream_t)stream);
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
    return launch_chain<MODE_FWD, ROLE_S>(tq, tk, tv, prm, (unsigned)p.frags.size(), (unsigned)p.H,
                                          (cudaStream_t)stream);
}

}  // namespace cpdr
