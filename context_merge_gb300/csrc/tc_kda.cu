// Per-dim gate (KDA) preparation for the tensor-core chains: the WY step of
// the article "flash-linear-attention 上下文并行CP ..." ([FLA-CP]) for a
// gate per key dimension.  §2.3: the per-dim Diag(alpha_t) is too costly
// inside the chunk recurrence, so the WY stage pre-gates the operands
// (kg = k 2^(g_last - g), qg = q 2^g) and the pre-process and the main
// kernel read the same gated tensors.  Per (chunk, head) unit, with
// G_i[d] = sum_{s <= i} g_s[d] / ln 2 inside the chunk and r = 31 the
// reference row of the factorised exponentials:
//   A_ij = beta_i sum_d k_id k_jd 2^(G_i[d] - G_j[d])      j < i
//   P_ij = sum_d q_id k_jd 2^(G_i[d] - G_j[d])             j <= i
//   T = (I + A)^-1;  T' = T diag(beta) (= T'': gamma lives in the tiles)
//   Kg = k 2^G, Kgam = k 2^(G_C - G) (bf16 hi, lo), Qg = q 2^G, gC = 2^(G_C)
// so that, in the chain, W = T' Kg, U = T' V, the state decays by Diag(gC)
// and takes Delta^T Kgam, and the output is (Qg) S + P Delta.
//
// A and P are sums of the factorised products (k 2^(G - G_r)) .
// (k 2^(G_r - G)) over the key dims, one 64 x 64 x 128 contraction each, on
// the tensor cores: the row operand X = [k 2^(G - G_r); q 2^(G - G_r)]
// (128 rows, A then P) goes into TMEM, the column operand F = k 2^(G_r - G)
// into shared memory, both split into bf16 hi and lo, and three products
// X_hi F_hi + X_lo F_hi + X_hi F_lo accumulate A and P in fp32 (the dropped
// lo . lo term is about 2^-16 of each product).  A unit whose in-chunk decay
// exceeds 2^100 either way of row r takes exact per-term exponentials on the
// CUDA cores instead.  One CTA per unit, two per SM: coalesced loads, column
// scans, the gated tiles, the operands, the products and their epilogue;
// then a second kernel solves T, a pair of warps per unit with the
// scalar-gate path's block solver, many units per SM at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"
#include "tc_gates.cuh"
#include "tc_solve.cuh"

namespace cpdr {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int C = 64;
constexpr int KP_THREADS = 256;
constexpr int KP_LD = D + 4;     // fp32 row stride of the [64][D] smem tiles
constexpr int kRef = 31;         // reference row of the factorised exponentials

struct KdaParams {
    const WyChunk *chunks;
    const __nv_bfloat16 *k, *q, *beta;
    const float *g;
    uint8_t *wy;
    uint8_t *qp;         // grouped query heads: Qg and P of query heads 1 .. G-1 of every unit
    int32_t *status;
    int H, G;            // state heads, query heads per state
};

// Shared memory (two CTAs per SM), from a 1 KiB-aligned base:
//   GF  [64][KP_LD] fp32: the gates, then G (log2 cumsum per key dim)
//   KB, QB [64][KQ_LD] bf16: k, q
//   FH, FL: hi and lo of k 2^(G_r - G) as two swizzled 64-column bf16
//           images each (the column operand of A and P)
// then beta, G_r, G_C, the steep flag, the MMA barrier, the abort flag and
// the TMEM slot.  At 101 KiB a preparation CTA cannot share an SM with a
// chain CTA (130 KiB or more), which holds all of TMEM.
constexpr int KQ_LD = D + 8;     // bf16 row stride (16-byte rows, offset banks)
constexpr int KP_OFF_KB = C * KP_LD * 4;
constexpr int KP_OFF_QB = KP_OFF_KB + C * KQ_LD * 2;
constexpr int KP_OFF_FH = (KP_OFF_QB + C * KQ_LD * 2 + 1023) & ~1023;
constexpr int KP_OFF_FL = KP_OFF_FH + 2 * 8192;
constexpr int KP_OFF_BETA = KP_OFF_FL + 2 * 8192;
constexpr int KP_OFF_GR = KP_OFF_BETA + C * 4;
constexpr int KP_OFF_GC = KP_OFF_GR + D * 4;
constexpr int KP_OFF_FLAG = KP_OFF_GC + D * 4;
constexpr int KP_OFF_BAR = KP_OFF_FLAG + 16;
constexpr int KP_OFF_CTL = KP_OFF_BAR + 16;
constexpr int KP_OFF_TSLOT = KP_OFF_CTL + 16;
constexpr size_t KP_SMEM = (size_t)KP_OFF_TSLOT + 16 + 1024;   // + alignment slack
static_assert(2 * (KP_SMEM + 1024) <= 233472, "two preparation CTAs must fit an SM");
static_assert(KP_SMEM + 1024 + (130 << 10) + 1024 > 233472, "a preparation CTA must not share an SM with a chain CTA");
// TMEM columns: X_hi [0, 64), X_lo [64, 128), the A / P accumulator [128, 192)
constexpr uint32_t KP_TMEM_COLS = 256;
constexpr uint32_t KP_COL_XLO = 64, KP_COL_ACC = 128;

// element (i, d) of a 64 x 128 bf16 tile stored as two swizzled 64-column images
__device__ __forceinline__ uint32_t img_off(int i, int d) {
    return (uint32_t)(d >> 6) * 8192u + sw128((uint32_t)i, (uint32_t)((d & 63) >> 3)) + (uint32_t)(d & 7) * 2u;
}
// 8 values as 8 bf16 (one 16-byte chunk)
__device__ __forceinline__ uint4 pack8f(const float *x) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
// hi = bf16(x) and lo = bf16(x - hi) of 8 values as 4 + 4 packed pairs
__device__ __forceinline__ void split8(const float *x, uint32_t *hi, uint32_t *lo) {
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        const float2 f = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x[2 * e] - f.x, x[2 * e + 1] - f.y);
        hi[e] = *reinterpret_cast<const uint32_t *>(&h);
        lo[e] = *reinterpret_cast<const uint32_t *>(&l);
    }
}
// the same, one 16-byte store each at byte offset `off` of the two images
__device__ __forceinline__ void store_hilo8(uint8_t *hi, uint8_t *lo, uint32_t off, const float *x) {
    uint32_t h[4], l[4];
    split8(x, h, l);
    *reinterpret_cast<uint4 *>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}
// 8 consecutive bf16 (one 16-byte chunk) as floats
__device__ __forceinline__ void unpack8(uint4 v, float *x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
// 16-byte asynchronous global-to-shared copy; `valid` false fills zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void ld8f(const float *p, float *x) {
    *reinterpret_cast<float4 *>(x) = *reinterpret_cast<const float4 *>(p);
    *reinterpret_cast<float4 *>(x + 4) = *reinterpret_cast<const float4 *>(p + 4);
}

// Exact exponentials per term (decays beyond 2^100 around row r), on the
// CUDA cores: A (strict lower, times beta; skipped when Ag is null) and P
// (lower including the diagonal, bf16 image at Pimg).  Thread (bi, bj) owns
// rows bi + 16 r and columns bj + 16 c (r, c < 4), so the column rows a warp
// reads are consecutive; pairs with j > i lie above the diagonal.
__device__ __noinline__ void exact_a_p(const float *GF, const __nv_bfloat16 *KB, const __nv_bfloat16 *QB,
                                       const float *beta, float *Ag, uint8_t *Pimg) {
    const int tid = threadIdx.x, bi = tid >> 4, bj = tid & 15;
    float a[4][4], pp[4][4];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 4; c++) a[r][c] = pp[r][c] = 0.f;
    for (int d = 0; d < D; d++) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int i = bi + 16 * r;
            const float Gi = GF[i * KP_LD + d], kv = __bfloat162float(KB[i * KQ_LD + d]);
            const float qv = __bfloat162float(QB[i * KQ_LD + d]);
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int j = bj + 16 * c;
                if (j > i) continue;
                const float lam = exp2f(Gi - GF[j * KP_LD + d]) * __bfloat162float(KB[j * KQ_LD + d]);
                a[r][c] = fmaf(kv, lam, a[r][c]);
                pp[r][c] = fmaf(qv, lam, pp[r][c]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; r++) {
        const int i = bi + 16 * r;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const int j = bj + 16 * c;
            if (Ag) Ag[i * C + j] = j < i ? beta[i] * a[r][c] : 0.f;
            *reinterpret_cast<__nv_bfloat16 *>(Pimg + sw128((uint32_t)i, (uint32_t)(j >> 3)) + (uint32_t)(j & 7) * 2u) =
                __float2bfloat16_rn(j <= i ? pp[r][c] : 0.f);
        }
    }
}

// GQA: the state has several query heads (a pass per query head); without
// it the single pass compiles to straight-line code.
template <bool GQA>
__global__ void __launch_bounds__(KP_THREADS, 2) tc_kda_prep_kernel(const __grid_constant__ KdaParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smb = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *GF = reinterpret_cast<float *>(smb);
    __nv_bfloat16 *KB = reinterpret_cast<__nv_bfloat16 *>(smb + KP_OFF_KB);
    __nv_bfloat16 *QB = reinterpret_cast<__nv_bfloat16 *>(smb + KP_OFF_QB);
    uint8_t *FH = smb + KP_OFF_FH, *FL = smb + KP_OFF_FL;
    float *beta = reinterpret_cast<float *>(smb + KP_OFF_BETA);
    float *Gr = reinterpret_cast<float *>(smb + KP_OFF_GR), *GCv = reinterpret_cast<float *>(smb + KP_OFF_GC);
    int *steep = reinterpret_cast<int *>(smb + KP_OFF_FLAG);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smb + KP_OFF_BAR);
    Ctl *ctl = reinterpret_cast<Ctl *>(smb + KP_OFF_CTL);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smb + KP_OFF_TSLOT);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, h = unit % p.H;
    const WyChunk ck = p.chunks[unit / p.H];
    const int nv = ck.nv;
    uint8_t *dst = p.wy + (size_t)unit * kKdaUnitBytes;
    auto tok = [&](int i) { return (ck.tok0 + i) * p.H + h; };
    // row i of query head gq of this state (q has G H heads)
    auto qtok = [&](int i, int gq) { return ((ck.tok0 + i) * p.H + h) * p.G + gq; };
    // Qg and P of query head gq: in the unit for the first, else in the
    // query-head region, laid out as in the unit
    auto qp_dst = [&](int gq) {
        return gq == 0 ? dst + kKdaOffQg : p.qp + ((size_t)unit * (p.G - 1) + (gq - 1)) * kKdaQpBytes;
    };

    if (tid == 0) {
        mbar_init(bar, 1);
        ctl->abort = 0;
        *steep = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 0) {
        tmem_alloc(tslot, KP_TMEM_COLS);
        tmem_relinquish();
    }

    // ---- loads: g, k, q of the chunk as 16-byte asynchronous copies, all in
    // flight at once (padded rows: zero-filled)
    {
        const uint32_t gf = smem_u32(GF), kb = smem_u32(KB), qb = smem_u32(QB);
#pragma unroll
        for (int m = 0; m < C * D / 4 / KP_THREADS; m++) {   // g: 32 copies per row
            const int e = tid + m * KP_THREADS, i = e >> 5, d = 4 * (e & 31);
            const int src = i < nv ? i : 0;
            cp_async16(gf + (uint32_t)(i * KP_LD + d) * 4u, p.g + (int64_t)tok(src) * D + d, i < nv);
        }
#pragma unroll
        for (int m = 0; m < C * D / 8 / KP_THREADS; m++) {   // k, q: 16 copies per row each
            const int e = tid + m * KP_THREADS, i = e >> 4, d = 8 * (e & 15);
            const int src = i < nv ? i : 0;
            cp_async16(kb + (uint32_t)(i * KQ_LD + d) * 2u, p.k + (int64_t)tok(src) * D + d, i < nv);
            cp_async16(qb + (uint32_t)(i * KQ_LD + d) * 2u, p.q + (int64_t)qtok(src, 0) * D + d, i < nv);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (tid < C) beta[tid] = tid < nv ? __bfloat162float(p.beta[tok(tid)]) : 0.f;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // ---- in-chunk cumulative log2 gates per key dim: two threads per column,
    // rows [0, 32) and [32, 64); the second half then adds the first's total
    {
        const int d = tid & (D - 1), h2 = tid >> 7;
        float run = 0.f;
        for (int i = 32 * h2; i < 32 * h2 + 32; i++) {
            run += GF[i * KP_LD + d] * kLog2e;
            GF[i * KP_LD + d] = run;
        }
        __syncthreads();
        const float gr = GF[kRef * KP_LD + d];   // the first half's total (kRef = 31)
        int far = 0;
        if (h2 == 1) {
            for (int i = 32; i < 64; i++) {
                const float x = GF[i * KP_LD + d] + gr;
                GF[i * KP_LD + d] = x;
                far |= fabsf(x - gr) > kFactorBound;
            }
            Gr[d] = gr;
            GCv[d] = GF[(C - 1) * KP_LD + d];
            reinterpret_cast<float *>(dst + kKdaOffGC)[d] = exp2f(GCv[d]);
        } else {
            for (int i = 0; i < 32; i++) far |= fabsf(GF[i * KP_LD + d] - gr) > kFactorBound;
        }
        if (__any_sync(0xffffffffu, far) && (tid & 31) == 0) atomicOr(steep, 1);
    }
    __syncthreads();
    const bool exact = *steep != 0;

    float *Ag = reinterpret_cast<float *>(dst);
    const int quad = w & 3, half = w >> 2;
    const int xr = 32 * quad + lane, xi = xr & 63;
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    // one pass per query head of this state (one without grouped query
    // heads): the first pass also builds the k tiles, F, X's k rows and A
    const int npass = GQA ? p.G : 1;
#pragma unroll 1
    for (int gq = 0; gq < npass; gq++) {
        const bool first = !GQA || gq == 0;
        uint8_t *qd = qp_dst(gq);
        if (!first) {
            // the previous pass's reads of QB and of the accumulator are done
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            const uint32_t qb = smem_u32(QB);
#pragma unroll
            for (int m = 0; m < C * D / 8 / KP_THREADS; m++) {
                const int e = tid + m * KP_THREADS, i = e >> 4, d = 8 * (e & 15);
                const int src = i < nv ? i : 0;
                cp_async16(qb + (uint32_t)(i * KQ_LD + d) * 2u, p.q + (int64_t)qtok(src, gq) * D + d, i < nv);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            __syncthreads();
        }

        // ---- gated tiles, and unless exact the column operand F (hi, lo).  A
        // thread takes 8 consecutive key dims of a row (one 16-byte chunk of
        // each image): items (row, group of 8), 4 per thread.
        if (first) {
            for (int item = tid; item < C * (D / 8); item += KP_THREADS) {
                const int i = item >> 4, d0 = (item & 15) * 8;
                float Gv[8], kv[8], qv[8], gc[8];
                ld8f(GF + i * KP_LD + d0, Gv);
                ld8f(GCv + d0, gc);
                unpack8(*reinterpret_cast<const uint4 *>(KB + i * KQ_LD + d0), kv);
                unpack8(*reinterpret_cast<const uint4 *>(QB + i * KQ_LD + d0), qv);
                float kg[8], kgam[8], qg[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const float gi = exp2f(Gv[e]);
                    kg[e] = kv[e] * gi;
                    kgam[e] = kv[e] * exp2f(gc[e] - Gv[e]);
                    qg[e] = qv[e] * gi;
                }
                const uint32_t off = img_off(i, d0);
                store_hilo8(dst + kKdaOffKg, dst + kKdaOffKgLo, off, kg);
                store_hilo8(dst + kKdaOffKgam, dst + kKdaOffKgamLo, off, kgam);
                *reinterpret_cast<uint4 *>(qd + off) = pack8f(qg);
                if (!exact) {
                    float gr[8], kf[8];
                    ld8f(Gr + d0, gr);
#pragma unroll
                    for (int e = 0; e < 8; e++) kf[e] = kv[e] * exp2f(gr[e] - Gv[e]);
                    store_hilo8(FH, FL, off, kf);
                }
            }
        } else {   // the query head's tile alone
            for (int item = tid; item < C * (D / 8); item += KP_THREADS) {
                const int i = item >> 4, d0 = (item & 15) * 8;
                float Gv[8], qv[8];
                ld8f(GF + i * KP_LD + d0, Gv);
                unpack8(*reinterpret_cast<const uint4 *>(QB + i * KQ_LD + d0), qv);
#pragma unroll
                for (int e = 0; e < 8; e++) qv[e] *= exp2f(Gv[e]);
                *reinterpret_cast<uint4 *>(qd + img_off(i, d0)) = pack8f(qv);
            }
        }

        // ---- the row operand X into TMEM: thread = one row of X (its warp's
        // lane quadrant: rows 0..63 the k rows of A, 64..127 the q rows of
        // P), half of the key dims per warp of a quadrant; lanes hold two K
        // elements per 32-bit column (lower key dim in the low half)
        if (!exact && (first || xr >= 64)) {
            const __nv_bfloat16 *src = xr < 64 ? KB : QB;
#pragma unroll
            for (int s = 0; s < 4; s++) {   // 16 key dims (8 columns) per step
                uint32_t hw[8], lw[8];
#pragma unroll
                for (int g2 = 0; g2 < 2; g2++) {
                    const int d0 = 64 * half + 16 * s + 8 * g2;
                    float Gv[8], gr[8], xv[8];
                    ld8f(GF + xi * KP_LD + d0, Gv);
                    ld8f(Gr + d0, gr);
                    unpack8(*reinterpret_cast<const uint4 *>(src + xi * KQ_LD + d0), xv);
#pragma unroll
                    for (int e = 0; e < 8; e++) xv[e] *= exp2f(Gv[e] - gr[e]);
                    split8(xv, hw + 4 * g2, lw + 4 * g2);
                }
                const uint32_t col = 32u * half + 8u * s;
                tmem_st8(trow + col, hw);
                tmem_st8(trow + KP_COL_XLO + col, lw);
            }
            tmem_st_wait();
        }
        fence_async_smem();   // F's stores become visible to the tensor core
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        if (!exact) {
            // ---- A and P (128 x 64, fp32 in TMEM) = X_hi F_hi + X_lo F_hi + X_hi F_lo
            if (tid == 0) {
                const uint32_t fh = smem_u32(FH), fl = smem_u32(FL);
                constexpr uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
                for (int pass = 0; pass < 3; pass++) {
                    const uint32_t xcol = pass == 1 ? KP_COL_XLO : 0u;
                    const uint32_t fb = pass == 2 ? fl : fh;
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++) {
                        const uint32_t koff = (uint32_t)(kk & 3) * 32u + (uint32_t)(kk >> 2) * 8192u;
                        mma_bf16_ts(tmem + KP_COL_ACC, tmem + xcol + 8u * kk, sdesc(fb + koff, 16, 1024), idesc,
                                    (pass | kk) != 0 ? 1u : 0u);
                    }
                }
                mma_commit(bar);
            }
            int ok = 0;
            if (lane == 0) ok = mbar_wait(bar, (uint32_t)(gq & 1), ctl, p.status, 120) ? 1 : 0;
            ok = __syncthreads_and(__shfl_sync(0xffffffffu, ok, 0));   // one verdict for the CTA
            if (ok) {
                tc_fence_after();
                const int j0 = 32 * half;
                if (xr < 64) {   // A row xi: strict lower part, times beta_i (first pass)
                    if (first) {
                        float vv[32];
                        tmem_ld32(trow + KP_COL_ACC + 32u * half, vv);
                        tmem_ld_wait();
                        const float bi = beta[xi];
#pragma unroll
                        for (int q4 = 0; q4 < 8; q4++) {
                            float4 a4;
                            const int j = j0 + 4 * q4;
                            a4.x = j < xi ? bi * vv[4 * q4] : 0.f;
                            a4.y = j + 1 < xi ? bi * vv[4 * q4 + 1] : 0.f;
                            a4.z = j + 2 < xi ? bi * vv[4 * q4 + 2] : 0.f;
                            a4.w = j + 3 < xi ? bi * vv[4 * q4 + 3] : 0.f;
                            *reinterpret_cast<float4 *>(Ag + xi * C + j) = a4;
                        }
                    }
                } else {         // P row xi: lower part including the diagonal
                    float vv[32];
                    tmem_ld32(trow + KP_COL_ACC + 32u * half, vv);
                    tmem_ld_wait();
#pragma unroll
                    for (int c8 = 0; c8 < 4; c8++) {
                        float pv[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) pv[e] = j0 + 8 * c8 + e <= xi ? vv[8 * c8 + e] : 0.f;
                        *reinterpret_cast<uint4 *>(qd + (kKdaOffP - kKdaOffQg) +
                                                   sw128((uint32_t)xi, (uint32_t)((j0 >> 3) + c8))) = pack8f(pv);
                    }
                }
            } else {
                if (lane == 0) {
                    // the products did not complete in time (status recorded):
                    // wait for them once more before the TMEM is released
                    Ctl local;
                    local.abort = 0;
                    mbar_wait(bar, (uint32_t)(gq & 1), &local, p.status, 121);
                }
                break;
            }
        } else {
            exact_a_p(GF, KB, QB, beta, first ? Ag : nullptr, qd + (kKdaOffP - kKdaOffQg));
        }
    }
    // A and beta go into the unit's first tiles, which the solve reads and
    // then overwrites with T', hi(T''), lo(T'')
    if (tid < C) reinterpret_cast<float *>(dst + 2 * kWyTileBytes)[tid] = beta[tid];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == 0) tmem_dealloc(tmem, KP_TMEM_COLS);
}

// T = (I + A)^-1 of every unit, a pair of warps per unit (persistent
// pairs, four per CTA, three CTAs per SM): A and beta from the unit (written
// above) into the pair's scratch, then the scalar-gate path's block solver
// overwrites the unit's first three tiles with T', hi(T''), lo(T'').
constexpr int KS_PAIRS = 4;
constexpr int KS_WARPS = 2 * KS_PAIRS;
constexpr size_t KS_SCRATCH = (size_t)C * kLS * 4 + 2 * C * 4;   // A, beta, ones
__global__ void __launch_bounds__(32 * KS_WARPS, 3) tc_kda_solve_kernel(uint8_t *wy, int n_units, float *tmat) {
    extern __shared__ __align__(16) uint8_t sms[];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pr = w >> 1, role = w & 1;
    const int bar_id = 1 + pr;   // named barrier of the pair
    float *S = reinterpret_cast<float *>(sms + pr * KS_SCRATCH);
    float *beta = S + C * kLS, *one = beta + C;
    if (role == 0) {
        one[lane] = 1.f;
        one[32 + lane] = 1.f;
    }
    for (int unit = blockIdx.x * KS_PAIRS + pr; unit < n_units; unit += gridDim.x * KS_PAIRS) {
        uint8_t *dst = wy + (size_t)unit * kKdaUnitBytes;
        const float4 *Ag = reinterpret_cast<const float4 *>(dst);
#pragma unroll 4
        for (int e = lane + 32 * role; e < C * C / 4; e += 64) {
            const int i = e / (C / 4), j = 4 * (e % (C / 4));
            *reinterpret_cast<float4 *>(S + i * kLS + j) = Ag[e];
        }
        if (role == 0) {
            const float *bg = reinterpret_cast<const float *>(dst + 2 * kWyTileBytes);
            beta[lane] = bg[lane];
            beta[32 + lane] = bg[32 + lane];
        }
        named_bar(bar_id, 64);   // A, beta (and the ones) in place; the unit's tiles read
        solve_unit_pair(S, dst, beta, one, role, bar_id, tmat ? tmat + (size_t)unit * C * C : nullptr);
        named_bar(bar_id, 64);   // the scratch has been read before the next unit's A
    }
}

}  // namespace

int launch_tc_kda_prep(const cpdr_ctx *c, const void *k, const void *q, const void *beta, const float *g,
                       void *wy, void *stream) {
    return launch_tc_kda_prep_t(c, k, q, beta, g, wy, nullptr, stream);
}

int launch_tc_kda_prep_t(const cpdr_ctx *c, const void *k, const void *q, const void *beta, const float *g,
                         void *wy, float *tmat, void *stream) {
    const auto &pl = c->plan;
    const int64_t units = (int64_t)pl.wy_chunks.size() * pl.H;
    if (units == 0) return 0;
    if (units > (int64_t)0x7fffffff) return (int)cudaErrorInvalidValue;
    KdaParams prm{};
    prm.chunks = c->dev.wy_chunks;
    prm.k = (const __nv_bfloat16 *)k;
    prm.q = (const __nv_bfloat16 *)q;
    prm.beta = (const __nv_bfloat16 *)beta;
    prm.g = g;
    prm.wy = (uint8_t *)wy;
    prm.qp = (uint8_t *)wy + (size_t)units * kKdaUnitBytes;
    prm.status = c->dev.status;
    prm.H = pl.H;
    prm.G = pl.G;
    auto kern = pl.G > 1 ? tc_kda_prep_kernel<true> : tc_kda_prep_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)KP_SMEM);
    if (e != cudaSuccess) return (int)e;
    kern<<<(unsigned)units, KP_THREADS, KP_SMEM, (cudaStream_t)stream>>>(prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    const size_t ssm = KS_PAIRS * KS_SCRATCH;   // one scratch per pair
    e = cudaFuncSetAttribute(tc_kda_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return (int)e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int64_t blocks = (units + KS_PAIRS - 1) / KS_PAIRS;
    const int grid = (int)std::min<int64_t>(blocks, (int64_t)sms * 3);
    tc_kda_solve_kernel<<<grid, 32 * KS_WARPS, ssm, (cudaStream_t)stream>>>((uint8_t *)wy, (int)units, tmat);
    return (int)cudaGetLastError();
}

}  // namespace cpdr
