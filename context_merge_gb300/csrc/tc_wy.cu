// WY build on the tensor-core path (bf16, d = 128, scalar gate): for every
// 64-token chunk of every fragment and every head ([FLA-CP] §2.2, the
// recompute_w_u step of its §4 Code Flow)
//   P  = K K^T                                          (tcgen05, fp32 in TMEM)
//   A  = beta_i 2^(G_i - G_j) P_ij, j < i               (SIMT)
//   T  = (I + A)^-1                                     (SIMT, fp32)
//   T' = T diag(beta),  T'' = T diag(beta gamma),  gamma_j = 2^(G_j)
// written as three bf16 64 x 64 tiles per (chunk, head): T', hi(T'') and
// lo(T'') = bf16(T'' - hi(T'')), each the 8 KiB 128-byte-swizzled image the
// chain kernels' MMAs read (K-major rows i, columns j).
//
// The solves of different chunks are independent, so they run here in one
// fully parallel launch; the chain kernels (tc_chain.cu) stream the tiles.
//
// CTA = 256 threads, two solve groups of four warps; one CTA iteration
// handles a pair of (chunk, head) units: one M = 128, N = 128 MMA computes
// [K_a; K_b][K_a; K_b]^T, whose diagonal blocks are K_a K_a^T (TMEM lanes and
// columns 0..63) and K_b K_b^T (lanes and columns 64..127).  Group 0 forms
// and inverts unit a, group 1 unit b.  The next pair's K tiles load while the
// groups solve.  Several CTAs share an SM (about 71 KB of shared memory,
// 128 TMEM columns each).  Waits are bounded as in the chain kernels.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"
#include "tc_gates.cuh"

namespace cpdr {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int WY_THREADS = 256;
constexpr int WY_CTAS_PER_SM = 3;
constexpr int kLS = 68;                           // scratch row stride (floats)
constexpr uint32_t WY_TMEM_COLS = 128;

// Shared-memory carve-up (byte offsets from a 1024-aligned base)
constexpr uint32_t O_KT = 0;                      // [a.c0 | b.c0 | a.c1 | b.c1], 8 KiB each
constexpr uint32_t O_SCR = 32768;                 // 2 groups x [64][68] fp32
constexpr uint32_t SCR_BYTES = 64 * kLS * 4;
constexpr int kWyGateFloats = 5 * 64 + 4;         // G, beta, gamma, e, f, flag
constexpr uint32_t O_GATES = O_SCR + 2 * SCR_BYTES;   // 2 groups x 2 slots
constexpr uint32_t O_BARS = O_GATES + 4 * kWyGateFloats * 4;
constexpr uint32_t O_CTL = O_BARS + 32;
constexpr uint32_t O_TSLOT = O_CTL + 16;
constexpr uint32_t WY_SMEM = O_TSLOT + 16;

struct WyParams {
    const WyChunk *chunks;
    const __nv_bfloat16 *beta;
    const float *g;
    uint8_t *wy;
    int32_t *status;
    int n_units;   // chunks x heads
    int H;
};

struct WyGates {
    float *G, *beta, *gam, *e, *f, *flag;
};
__device__ __forceinline__ WyGates wy_gates(uint8_t *base, int group, int slot) {
    float *q = reinterpret_cast<float *>(base + O_GATES) + (2 * group + slot) * kWyGateFloats;
    return WyGates{q, q + 64, q + 128, q + 192, q + 256, q + 320};
}

// Writes T' = T diag(beta), hi(T'') and lo(T'') for 4 consecutive columns
// j0.. of row i into the unit's three tiles in global memory.
__device__ __forceinline__ void put_t4(uint8_t *dst, const WyGates &gs, int i, int j0, float t0, float t1,
                                       float t2, float t3) {
    const float4 b4 = *reinterpret_cast<const float4 *>(gs.beta + j0);
    const float4 g4 = *reinterpret_cast<const float4 *>(gs.gam + j0);
    const float a0 = t0 * b4.x, a1 = t1 * b4.y, a2 = t2 * b4.z, a3 = t3 * b4.w;
    const float c0 = a0 * g4.x, c1 = a1 * g4.y, c2 = a2 * g4.z, c3 = a3 * g4.w;
    const uint32_t off = sw128(i, j0 >> 3) + (j0 & 4) * 2;
    uint2 u, hi, lo;
    u.x = pack_bf16(a0, a1);
    u.y = pack_bf16(a2, a3);
    hi.x = pack_bf16(c0, c1);
    hi.y = pack_bf16(c2, c3);
    const float2 h01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi.x));
    const float2 h23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi.y));
    lo.x = pack_bf16(c0 - h01.x, c1 - h01.y);
    lo.y = pack_bf16(c2 - h23.x, c3 - h23.y);
    *reinterpret_cast<uint2 *>(dst + off) = u;
    *reinterpret_cast<uint2 *>(dst + kWyTileBytes + off) = hi;
    *reinterpret_cast<uint2 *>(dst + 2 * kWyTileBytes + off) = lo;
}

// In-place inverse T = (I + A)^-1 of the unit lower-triangular matrix held
// in S[64][68] (strictly lower part = A, the rest 0), 128 threads of named
// barrier `bar`, and the tiles written from it:
//   1. the four 16x16 diagonal blocks by forward substitution (row-prefetched);
//   2. inside each 32x32 diagonal block: X21 = -T22 (A21 T11)  (16x16 blocks);
//   3. the 64x64 level:               X21 = -T22 (A21 T11)  (32x32 blocks).
// Each product is computed into registers and written back after a barrier.
// The tiles of the two 32x32 diagonal blocks are written during step 3's
// first product, those of the off-diagonal block straight from registers.
__device__ __forceinline__ void solve_inverse(float *S, uint8_t *dst, const WyGates &gs, int t, int bar) {
    // 1. diagonal 16x16 blocks: thread (b, col), t < 64.  x_i = -sum_k A[i][k] x_k
    //    over the whole row (the row is zero from k = i on, x is zero before col).
    {
        float x[16];
        const int b = t >> 4, col = t & 15;
        if (t < 64) {
            const float *Ab = S + (16 * b) * kLS + 16 * b;
#pragma unroll
            for (int i = 0; i < 16; i++) x[i] = 0.f;
            float4 nxt[4];
#pragma unroll
            for (int q = 0; q < 4; q++) nxt[q] = *reinterpret_cast<const float4 *>(Ab + 4 * q);
#pragma unroll
            for (int i = 0; i < 16; i++) {
                float4 row[4];
#pragma unroll
                for (int q = 0; q < 4; q++) row[q] = nxt[q];
                if (i + 1 < 16) {
#pragma unroll
                    for (int q = 0; q < 4; q++) nxt[q] = *reinterpret_cast<const float4 *>(Ab + (i + 1) * kLS + 4 * q);
                }
                float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    if (4 * q < i) {
                        p0 = fmaf(row[q].x, x[4 * q], p0);
                        p1 = fmaf(row[q].y, x[4 * q + 1], p1);
                        p2 = fmaf(row[q].z, x[4 * q + 2], p2);
                        p3 = fmaf(row[q].w, x[4 * q + 3], p3);
                    }
                }
                const float sum = (p0 + p1) + (p2 + p3);
                x[i] = (i < col) ? 0.f : (i == col ? 1.f : -sum);
            }
        }
        named_bar(bar, 128);
        if (t < 64) {
            float *Ab = S + (16 * b) * kLS + 16 * b;
#pragma unroll
            for (int i = 0; i < 16; i++) Ab[i * kLS + col] = x[i];
        }
        named_bar(bar, 128);
    }
    // 2. 16x16 off-diagonal blocks of the two 32x32 diagonal blocks:
    //    thread (p, i, 4 columns): rows 32p + 16 + i, columns 32p + jq ..
    {
        const int p = t >> 6, i = (t & 63) >> 2, jq = (t & 3) * 4;
        const int r1 = 32 * p + 16, c0 = 32 * p;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 16; k++) {   // Y = A21 T11
            const float a = S[(r1 + i) * kLS + c0 + k];
            const float4 tr = *reinterpret_cast<const float4 *>(S + (c0 + k) * kLS + c0 + jq);
            y[0] = fmaf(a, tr.x, y[0]); y[1] = fmaf(a, tr.y, y[1]);
            y[2] = fmaf(a, tr.z, y[2]); y[3] = fmaf(a, tr.w, y[3]);
        }
        named_bar(bar, 128);
        *reinterpret_cast<float4 *>(S + (r1 + i) * kLS + c0 + jq) = make_float4(y[0], y[1], y[2], y[3]);
        named_bar(bar, 128);
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 16; k++) {   // X = -T22 Y
            const float a = S[(r1 + i) * kLS + r1 + k];
            const float4 yr = *reinterpret_cast<const float4 *>(S + (r1 + k) * kLS + c0 + jq);
            x[0] = fmaf(a, yr.x, x[0]); x[1] = fmaf(a, yr.y, x[1]);
            x[2] = fmaf(a, yr.z, x[2]); x[3] = fmaf(a, yr.w, x[3]);
        }
        named_bar(bar, 128);
        *reinterpret_cast<float4 *>(S + (r1 + i) * kLS + c0 + jq) = make_float4(-x[0], -x[1], -x[2], -x[3]);
        named_bar(bar, 128);
    }
    // 3. the 32x32 off-diagonal block (rows 32..63, columns 0..31): thread (i, 8 columns)
    {
        const int i = t >> 2, jo = (t & 3) * 8;
        float y[8];
#pragma unroll
        for (int u = 0; u < 8; u++) y[u] = 0.f;
        float an = S[(32 + i) * kLS];
        float4 t0n = *reinterpret_cast<const float4 *>(S + jo), t1n = *reinterpret_cast<const float4 *>(S + jo + 4);
#pragma unroll
        for (int k = 0; k < 32; k++) {   // Y = A21 T11 (operands of k+1 loaded ahead)
            const float a = an;
            const float4 t0 = t0n, t1 = t1n;
            if (k + 1 < 32) {
                an = S[(32 + i) * kLS + k + 1];
                t0n = *reinterpret_cast<const float4 *>(S + (k + 1) * kLS + jo);
                t1n = *reinterpret_cast<const float4 *>(S + (k + 1) * kLS + jo + 4);
            }
            y[0] = fmaf(a, t0.x, y[0]); y[1] = fmaf(a, t0.y, y[1]); y[2] = fmaf(a, t0.z, y[2]);
            y[3] = fmaf(a, t0.w, y[3]); y[4] = fmaf(a, t1.x, y[4]); y[5] = fmaf(a, t1.y, y[5]);
            y[6] = fmaf(a, t1.z, y[6]); y[7] = fmaf(a, t1.w, y[7]);
        }
        // the two 32x32 diagonal blocks of T are final: write their tiles
        // (thread (i, 8 columns) of each block)
#pragma unroll
        for (int blk = 0; blk < 2; blk++) {
            const int ii = 32 * blk + i, jj = 32 * blk + jo;
            const float4 v0 = *reinterpret_cast<const float4 *>(S + ii * kLS + jj);
            const float4 v1 = *reinterpret_cast<const float4 *>(S + ii * kLS + jj + 4);
            put_t4(dst, gs, ii, jj, v0.x, v0.y, v0.z, v0.w);
            put_t4(dst, gs, ii, jj + 4, v1.x, v1.y, v1.z, v1.w);
        }
        // the zero upper-right block (rows 0..31, columns 32..63)
        put_t4(dst, gs, i, 32 + jo, 0.f, 0.f, 0.f, 0.f);
        put_t4(dst, gs, i, 32 + jo + 4, 0.f, 0.f, 0.f, 0.f);
        named_bar(bar, 128);
        *reinterpret_cast<float4 *>(S + (32 + i) * kLS + jo) = make_float4(y[0], y[1], y[2], y[3]);
        *reinterpret_cast<float4 *>(S + (32 + i) * kLS + jo + 4) = make_float4(y[4], y[5], y[6], y[7]);
        named_bar(bar, 128);
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; u++) x[u] = 0.f;
        an = S[(32 + i) * kLS + 32];
        t0n = *reinterpret_cast<const float4 *>(S + 32 * kLS + jo);
        t1n = *reinterpret_cast<const float4 *>(S + 32 * kLS + jo + 4);
#pragma unroll
        for (int k = 0; k < 32; k++) {   // X = -T22 Y (operands of k+1 loaded ahead)
            const float a = an;
            const float4 t0 = t0n, t1 = t1n;
            if (k + 1 < 32) {
                an = S[(32 + i) * kLS + 32 + k + 1];
                t0n = *reinterpret_cast<const float4 *>(S + (32 + k + 1) * kLS + jo);
                t1n = *reinterpret_cast<const float4 *>(S + (32 + k + 1) * kLS + jo + 4);
            }
            x[0] = fmaf(a, t0.x, x[0]); x[1] = fmaf(a, t0.y, x[1]); x[2] = fmaf(a, t0.z, x[2]);
            x[3] = fmaf(a, t0.w, x[3]); x[4] = fmaf(a, t1.x, x[4]); x[5] = fmaf(a, t1.y, x[5]);
            x[6] = fmaf(a, t1.z, x[6]); x[7] = fmaf(a, t1.w, x[7]);
        }
        // the off-diagonal block's tiles straight from registers
        put_t4(dst, gs, 32 + i, jo, -x[0], -x[1], -x[2], -x[3]);
        put_t4(dst, gs, 32 + i, jo + 4, -x[4], -x[5], -x[6], -x[7]);
    }
}

// Warp-uniform bounded wait (lane 0 polls, the verdict is broadcast).
__device__ __forceinline__ bool wy_warp_wait(uint64_t *bar, uint32_t parity, Ctl *ctl, int32_t *status, int site) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, ctl, status, site) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

__global__ void __launch_bounds__(WY_THREADS, WY_CTAS_PER_SM)
tc_wy_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ WyParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int grp = tid >> 7, t = tid & 127;
    // [0] K tiles landed, [1] P ready, [2] drain
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + O_BARS);
    Ctl *ctl = reinterpret_cast<Ctl *>(base + O_CTL);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + O_TSLOT);
    const int npairs = (p.n_units + 1) >> 1;
    const int H = p.H;

    // loads the K tiles of pair q (a: rows 0..63, b: rows 64..127 of the stacked tile)
    auto issue_pair = [&](int q) {
        const int ua = 2 * q, ub = 2 * q + 1;
        const bool has_b = ub < p.n_units;
        mbar_arrive_expect_tx(&bar[0], has_b ? 32768u : 16384u);
        const int ha = ua % H, tok_a = (int)p.chunks[ua / H].tok0;
        tma_load_3d(base + O_KT, &tk, &bar[0], 0, ha, tok_a);
        tma_load_3d(base + O_KT + 16384, &tk, &bar[0], 64, ha, tok_a);
        if (has_b) {
            const int hb = ub % H, tok_b = (int)p.chunks[ub / H].tok0;
            tma_load_3d(base + O_KT + 8192, &tk, &bar[0], 0, hb, tok_b);
            tma_load_3d(base + O_KT + 24576, &tk, &bar[0], 64, hb, tok_b);
        }
    };

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tk);
    }
    if (w == 0) {
        tmem_alloc(tslot, WY_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    int issued = -1;   // iteration whose K load is in flight
    if (tid == 0 && (int)blockIdx.x < npairs) {
        issue_pair(blockIdx.x);
        issued = 0;
    }
    const uint32_t b0 = smem_u32(base);
    const uint64_t d_kt = sdesc(b0 + O_KT, 16, 1024);
    int it = 0;
    for (int q = blockIdx.x; q < npairs; q += gridDim.x, it++) {
        const int unit = 2 * q + grp;
        const bool valid = unit < p.n_units;
        const WyGates gs = wy_gates(base, grp, it & 1);
        // P = [K_a; K_b][K_a; K_b]^T
        if (tid == 0) {
            if (mbar_wait(&bar[0], it & 1, ctl, p.status, 80)) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint64_t o = (uint64_t)(((k & 3) * 32 + (k >> 2) * 16384) >> 4);
                    mma_bf16(tmem, d_kt + o, d_kt + o, idesc_bf16(128, 128, false, false), k > 0 ? 1u : 0u);
                }
                mma_commit(&bar[1]);
            }
        }
        // gates of this group's unit (warp 0 of the group; padded rows: 0)
        if ((w & 3) == 0 && valid) {
            const WyChunk ck = p.chunks[unit / H];
            const int h = unit % H;
            const int i0 = 2 * lane, i1 = 2 * lane + 1;
            float b0v = 0.f, b1v = 0.f, g0 = 0.f, g1 = 0.f;
            if (i0 < ck.nv) {
                b0v = __bfloat162float(p.beta[(ck.tok0 + i0) * H + h]);
                g0 = p.g[(ck.tok0 + i0) * H + h] * kLog2e;
            }
            if (i1 < ck.nv) {
                b1v = __bfloat162float(p.beta[(ck.tok0 + i1) * H + h]);
                g1 = p.g[(ck.tok0 + i1) * H + h] * kLog2e;
            }
            const LaneGates lg = scan_gates(g0, g1);
            gs.G[i0] = lg.G0; gs.G[i1] = lg.G1;
            gs.beta[i0] = b0v; gs.beta[i1] = b1v;
            gs.gam[i0] = exp2f(lg.G0); gs.gam[i1] = exp2f(lg.G1);
            gs.e[i0] = exp2f(lg.G0 - lg.Gr); gs.e[i1] = exp2f(lg.G1 - lg.Gr);
            gs.f[i0] = exp2f(lg.Gr - lg.G0); gs.f[i1] = exp2f(lg.Gr - lg.G1);
            if (lane == 0) gs.flag[0] = lg.exact ? 1.f : 0.f;
        }
        const bool pok = wy_warp_wait(&bar[1], it & 1, ctl, p.status, 81);
        __syncthreads();   // gates published; the verdicts of both waits are in ctl->abort
        if (ctl->abort || !pok) break;
        tc_fence_after();
        float *S = reinterpret_cast<float *>(base + O_SCR + grp * SCR_BYTES);
        // A rows from TMEM: group 0 -> warps 0, 1 (lanes 0..63, columns 0..63),
        // group 1 -> warps 6, 7 (lanes 64..127, columns 64..127)
        const int wq = w & 3;
        if (valid && (wq >> 1) == grp) {
            const int i = 32 * (wq & 1) + lane;
            const bool exact = gs.flag[0] != 0.f;
            const float bi = gs.beta[i], Gi = gs.G[i], bei = gs.beta[i] * gs.e[i];
#pragma unroll
            for (int half = 0; half < 2; half++) {
                float vv[32];
                tmem_ld32(tmem + ((uint32_t)(32 * wq) << 16) + 64 * grp + 32 * half, vv);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 8; q4++) {
                    const int j0 = 32 * half + 4 * q4;
                    const float4 f4 = *reinterpret_cast<const float4 *>(gs.f + j0);
                    const float fv[4] = {f4.x, f4.y, f4.z, f4.w};
                    float e4[4];
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const float x = vv[4 * q4 + u];
                        const float val = exact ? bi * exp2f(Gi - gs.G[j0 + u]) * x : bei * fv[u] * x;
                        e4[u] = (j0 + u < i) ? val : 0.f;
                    }
                    *reinterpret_cast<float4 *>(S + i * kLS + j0) = make_float4(e4[0], e4[1], e4[2], e4[3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();   // TMEM read and the K tiles consumed: load the next pair
        if (tid == 0) {
            const int qn = q + gridDim.x;
            if (qn < npairs) {
                issue_pair(qn);
                issued = it + 1;
            }
        }
        if (valid) {
            uint8_t *dst = p.wy + (size_t)unit * kWyUnitBytes;
            solve_inverse(S, dst, gs, t, 1 + grp);
        }
    }
    // every issued load and MMA must have completed before the CTA exits
    if (tid == 0) {
        Ctl local;
        local.abort = 0;
        if (issued >= it) mbar_wait(&bar[0], issued & 1, &local, p.status, 82);
        mma_commit(&bar[2]);
        mbar_wait(&bar[2], 0, &local, p.status, 83);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == 0) tmem_dealloc(tmem, WY_TMEM_COLS);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn wy_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

}  // namespace

size_t wy_bytes(const cpdr_ctx *c) {
    if (!c->use_tc) return 0;
    return c->plan.wy_chunks.size() * (size_t)c->plan.H * kWyUnitBytes;
}

int launch_tc_wy(const cpdr_ctx *c, const void *k, const void *beta, const float *g, void *wy, void *stream) {
    const auto &pl = c->plan;
    const int64_t units = (int64_t)pl.wy_chunks.size() * pl.H;
    if (units == 0) return 0;
    if (units > (int64_t)0x7fffffff) return (int)cudaErrorInvalidValue;
    EncodeTiledFn fn = wy_encode_fn();
    if (!fn) return (int)cudaErrorInvalidValue;
    // k as [B*T, H, D] bf16, box {64, 1, 64}, 128-byte swizzle (the chain kernels' map)
    CUtensorMap tk;
    const int64_t tokens = (int64_t)pl.B * pl.T;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pl.H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)pl.H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(k), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return (int)cudaErrorInvalidValue;
    WyParams prm{};
    prm.chunks = c->dev.wy_chunks;
    prm.beta = (const __nv_bfloat16 *)beta;
    prm.g = g;
    prm.wy = (uint8_t *)wy;
    prm.status = c->dev.status;
    prm.n_units = (int)units;
    prm.H = pl.H;
    const size_t smem = WY_SMEM + 1024;
    cudaError_t e = cudaFuncSetAttribute(tc_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int npairs = (int)((units + 1) / 2);
    const int grid = npairs < sms * WY_CTAS_PER_SM ? npairs : sms * WY_CTAS_PER_SM;
    tc_wy_kernel<<<grid, WY_THREADS, smem, (cudaStream_t)stream>>>(tk, prm);
    return (int)cudaGetLastError();
}

}  // namespace cpdr
