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
// A and P are fp32 sums of the factorised products (k 2^(G - G_r)) .
// (k 2^(G_r - G)) (the q factor rounded to bf16: P is a bf16 tile); a unit
// whose in-chunk decay exceeds 2^100 either way of row r takes exact
// per-term exponentials instead.  One CTA per unit, two per SM (CUDA
// cores): coalesced loads, column scans, the gated tiles, A and P; then a
// second kernel solves T, one warp per unit with the scalar-gate path's
// solver, many units per SM at once.
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
    int H;
};

// Shared memory (two CTAs per SM):
//   GF  [64][KP_LD] fp32: G (log2 cumsum), then k 2^(G_r - G)      ("KF")
//   KB  [64][KP_LD] fp32: k, then k 2^(G - G_r)                     ("KE")
//   QB  [64][KQ_LD] bf16: q, then bf16(q 2^(G - G_r))
// then beta, G_r, G_C and the steep flag.
constexpr int KQ_LD = D + 8;     // bf16 row stride (16-byte rows, offset banks)
constexpr int KP_OFF_KB = C * KP_LD * 4;
constexpr int KP_OFF_QB = 2 * C * KP_LD * 4;
constexpr int KP_OFF_BETA = KP_OFF_QB + C * KQ_LD * 2;
constexpr int KP_OFF_GR = KP_OFF_BETA + C * 4;
constexpr int KP_OFF_GC = KP_OFF_GR + D * 4;
constexpr int KP_OFF_FLAG = KP_OFF_GC + D * 4;
constexpr size_t KP_SMEM = (size_t)KP_OFF_FLAG + 16;
static_assert(2 * (KP_SMEM + 1024) <= 233472, "two preparation CTAs must fit an SM");

// element (i, d) of a 64 x 128 bf16 tile stored as two swizzled 64-column images
__device__ __forceinline__ uint32_t img_off(int i, int d) {
    return (uint32_t)(d >> 6) * 8192u + sw128((uint32_t)i, (uint32_t)((d & 63) >> 3)) + (uint32_t)(d & 7) * 2u;
}
__device__ __forceinline__ void put_bf16(uint8_t *img, uint32_t off, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(img + off) = __float2bfloat16_rn(x);
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
// hi = bf16(x) and lo = bf16(x - hi) of 8 values, one 16-byte store each
__device__ __forceinline__ void store_hilo8(uint8_t *hi, uint8_t *lo, uint32_t off, const float *x, uint4 &h) {
    h = pack8f(x);
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
    float r[8];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hw[e]));
        r[2 * e] = x[2 * e] - f.x;
        r[2 * e + 1] = x[2 * e + 1] - f.y;
    }
    *reinterpret_cast<uint4 *>(hi + off) = h;
    *reinterpret_cast<uint4 *>(lo + off) = pack8f(r);
}

__global__ void __launch_bounds__(KP_THREADS, 2) tc_kda_prep_kernel(const __grid_constant__ KdaParams p) {
    extern __shared__ __align__(16) uint8_t smb[];
    float *GF = reinterpret_cast<float *>(smb);
    float *KB = reinterpret_cast<float *>(smb + KP_OFF_KB);
    __nv_bfloat16 *QB = reinterpret_cast<__nv_bfloat16 *>(smb + KP_OFF_QB);
    float *beta = reinterpret_cast<float *>(smb + KP_OFF_BETA);
    float *Gr = reinterpret_cast<float *>(smb + KP_OFF_GR), *GCv = reinterpret_cast<float *>(smb + KP_OFF_GC);
    int *steep = reinterpret_cast<int *>(smb + KP_OFF_FLAG);
    const int tid = threadIdx.x;
    const int unit = blockIdx.x, h = unit % p.H;
    const WyChunk ck = p.chunks[unit / p.H];
    const int nv = ck.nv;
    uint8_t *dst = p.wy + (size_t)unit * kKdaUnitBytes;
    auto tok = [&](int i) { return (ck.tok0 + i) * p.H + h; };

    // ---- loads: g, k, q of the chunk (padded rows: 0), every load independent
    for (int e = tid; e < C * D / 4; e += KP_THREADS) {
        const int i = e / (D / 4), d = 4 * (e % (D / 4));
        float4 g4 = make_float4(0.f, 0.f, 0.f, 0.f);
        uint2 k2 = make_uint2(0u, 0u), q2 = make_uint2(0u, 0u);
        if (i < nv) {
            g4 = __ldg(reinterpret_cast<const float4 *>(p.g + (int64_t)tok(i) * D + d));
            k2 = __ldg(reinterpret_cast<const uint2 *>(p.k + (int64_t)tok(i) * D + d));
            q2 = __ldg(reinterpret_cast<const uint2 *>(p.q + (int64_t)tok(i) * D + d));
        }
        *reinterpret_cast<float4 *>(GF + i * KP_LD + d) = g4;
        const float2 ka = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&k2.x));
        const float2 kb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&k2.y));
        *reinterpret_cast<float4 *>(KB + i * KP_LD + d) = make_float4(ka.x, ka.y, kb.x, kb.y);
        *reinterpret_cast<uint2 *>(QB + i * KQ_LD + d) = q2;
    }
    if (tid < C) beta[tid] = tid < nv ? __bfloat162float(p.beta[tok(tid)]) : 0.f;
    if (tid == 0) *steep = 0;
    __syncthreads();

    // ---- in-chunk cumulative log2 gates per key dim
    if (tid < D) {
        float run = 0.f;
        int far = 0;
        for (int i = 0; i < C; i++) {
            run += GF[i * KP_LD + tid] * kLog2e;
            GF[i * KP_LD + tid] = run;
        }
        const float gr = GF[kRef * KP_LD + tid];
        for (int i = 0; i < C; i++) far |= fabsf(GF[i * KP_LD + tid] - gr) > kFactorBound;
        Gr[tid] = gr;
        GCv[tid] = run;
        reinterpret_cast<float *>(dst + kKdaOffGC)[tid] = exp2f(run);
        if (__any_sync(0xffffffffu, far) && (tid & 31) == 0) atomicOr(steep, 1);
    }
    __syncthreads();
    const bool exact = *steep != 0;

    // ---- gated tiles; unless exact, the factorised operands replace the
    // inputs in place.  A thread takes 8 consecutive key dims of a row (one
    // 16-byte chunk of each image): items (row, group of 8), 4 per thread.
    for (int item = tid; item < C * (D / 8); item += KP_THREADS) {
        const int i = item >> 4, d0 = (item & 15) * 8;
        float Gv[8], kv[8], qv[8], gr[8], gc[8];
        *reinterpret_cast<float4 *>(Gv) = *reinterpret_cast<const float4 *>(GF + i * KP_LD + d0);
        *reinterpret_cast<float4 *>(Gv + 4) = *reinterpret_cast<const float4 *>(GF + i * KP_LD + d0 + 4);
        *reinterpret_cast<float4 *>(kv) = *reinterpret_cast<const float4 *>(KB + i * KP_LD + d0);
        *reinterpret_cast<float4 *>(kv + 4) = *reinterpret_cast<const float4 *>(KB + i * KP_LD + d0 + 4);
        *reinterpret_cast<float4 *>(gr) = *reinterpret_cast<const float4 *>(Gr + d0);
        *reinterpret_cast<float4 *>(gr + 4) = *reinterpret_cast<const float4 *>(Gr + d0 + 4);
        *reinterpret_cast<float4 *>(gc) = *reinterpret_cast<const float4 *>(GCv + d0);
        *reinterpret_cast<float4 *>(gc + 4) = *reinterpret_cast<const float4 *>(GCv + d0 + 4);
        {
            const uint4 q8 = *reinterpret_cast<const uint4 *>(QB + i * KQ_LD + d0);
            const uint32_t qw[4] = {q8.x, q8.y, q8.z, q8.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qw[e]));
                qv[2 * e] = f.x;
                qv[2 * e + 1] = f.y;
            }
        }
        float kg[8], kgam[8], qg[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const float gi = exp2f(Gv[e]);
            kg[e] = kv[e] * gi;
            kgam[e] = kv[e] * exp2f(gc[e] - Gv[e]);
            qg[e] = qv[e] * gi;
        }
        const uint32_t off = img_off(i, d0);
        uint4 h_kg, h_kgam;
        store_hilo8(dst + kKdaOffKg, dst + kKdaOffKgLo, off, kg, h_kg);
        store_hilo8(dst + kKdaOffKgam, dst + kKdaOffKgamLo, off, kgam, h_kgam);
        *reinterpret_cast<uint4 *>(dst + kKdaOffQg + off) = pack8f(qg);
        if (!exact) {
            float ke[8], kf[8], qe[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const float ef = exp2f(Gv[e] - gr[e]);
                ke[e] = kv[e] * ef;
                kf[e] = kv[e] * exp2f(gr[e] - Gv[e]);
                qe[e] = qv[e] * ef;
            }
            *reinterpret_cast<float4 *>(GF + i * KP_LD + d0) = *reinterpret_cast<const float4 *>(kf);
            *reinterpret_cast<float4 *>(GF + i * KP_LD + d0 + 4) = *reinterpret_cast<const float4 *>(kf + 4);
            *reinterpret_cast<float4 *>(KB + i * KP_LD + d0) = *reinterpret_cast<const float4 *>(ke);
            *reinterpret_cast<float4 *>(KB + i * KP_LD + d0 + 4) = *reinterpret_cast<const float4 *>(ke + 4);
            *reinterpret_cast<uint4 *>(QB + i * KQ_LD + d0) = pack8f(qe);
        }
    }
    __syncthreads();

    // ---- A (strict lower, times beta_i) and P (lower incl. the diagonal):
    // thread (bi, bj) owns rows bi + 16 r and columns bj + 16 c (r, c < 4),
    // so the 16 column rows a warp reads are consecutive (no bank conflicts);
    // pairs with c > r lie above the diagonal and are skipped
    const int bi = tid >> 4, bj = tid & 15;
    float a[4][4], pp[4][4];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 4; c++) a[r][c] = pp[r][c] = 0.f;
    if (!exact) {
        for (int d = 0; d < D; d += 4) {
            float4 ke[4], kf[4];
            float qe[4][4];
#pragma unroll
            for (int r = 0; r < 4; r++) {
                ke[r] = *reinterpret_cast<const float4 *>(KB + (bi + 16 * r) * KP_LD + d);
                kf[r] = *reinterpret_cast<const float4 *>(GF + (bj + 16 * r) * KP_LD + d);
                const uint2 q2 = *reinterpret_cast<const uint2 *>(QB + (bi + 16 * r) * KQ_LD + d);
                const float2 qa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q2.x));
                const float2 qb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q2.y));
                qe[r][0] = qa.x; qe[r][1] = qa.y; qe[r][2] = qb.x; qe[r][3] = qb.y;
            }
#pragma unroll
            for (int r = 0; r < 4; r++)
#pragma unroll
                for (int c = 0; c <= r; c++) {   // column block c > r lies above the diagonal
                    a[r][c] = fmaf(ke[r].x, kf[c].x, a[r][c]);
                    a[r][c] = fmaf(ke[r].y, kf[c].y, a[r][c]);
                    a[r][c] = fmaf(ke[r].z, kf[c].z, a[r][c]);
                    a[r][c] = fmaf(ke[r].w, kf[c].w, a[r][c]);
                    pp[r][c] = fmaf(qe[r][0], kf[c].x, pp[r][c]);
                    pp[r][c] = fmaf(qe[r][1], kf[c].y, pp[r][c]);
                    pp[r][c] = fmaf(qe[r][2], kf[c].z, pp[r][c]);
                    pp[r][c] = fmaf(qe[r][3], kf[c].w, pp[r][c]);
                }
        }
    } else {
        // exact exponentials per term (decays beyond 2^100 around row r)
        for (int d = 0; d < D; d++) {
#pragma unroll
            for (int r = 0; r < 4; r++) {
                const int i = bi + 16 * r;
                const float Gi = GF[i * KP_LD + d], kv = KB[i * KP_LD + d];
                const float qv = __bfloat162float(QB[i * KQ_LD + d]);
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int j = bj + 16 * c;
                    if (j > i) continue;
                    const float lam = exp2f(Gi - GF[j * KP_LD + d]) * KB[j * KP_LD + d];
                    a[r][c] = fmaf(kv, lam, a[r][c]);
                    pp[r][c] = fmaf(qv, lam, pp[r][c]);
                }
            }
        }
    }
    // A (fp32, row-major 64 x 64) and beta go into the unit's first tiles,
    // which the solve reads and then overwrites with T', hi(T''), lo(T'')
    float *Ag = reinterpret_cast<float *>(dst);
#pragma unroll
    for (int r = 0; r < 4; r++) {
        const int i = bi + 16 * r;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const int j = bj + 16 * c;
            Ag[i * C + j] = j < i ? beta[i] * a[r][c] : 0.f;
            put_bf16(dst + kKdaOffP, sw128((uint32_t)i, (uint32_t)(j >> 3)) + (uint32_t)(j & 7) * 2u,
                     j <= i ? pp[r][c] : 0.f);
        }
    }
    if (tid < C) reinterpret_cast<float *>(dst + 2 * kWyTileBytes)[tid] = beta[tid];
}

// T = (I + A)^-1 of every unit, one warp per unit (persistent warps): A and
// beta from the unit (written above) into this warp's scratch, then the
// solver overwrites the unit's first three tiles with T', hi(T''), lo(T'').
constexpr int KS_WARPS = 4;
constexpr size_t KS_SCRATCH = (size_t)C * kLS * 4 + 2 * C * 4;   // A, beta, ones
__global__ void __launch_bounds__(32 * KS_WARPS) tc_kda_solve_kernel(uint8_t *wy, int n_units) {
    extern __shared__ __align__(16) uint8_t sms[];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *S = reinterpret_cast<float *>(sms + w * KS_SCRATCH);
    float *beta = S + C * kLS, *one = beta + C;
    one[lane] = 1.f;
    one[32 + lane] = 1.f;
    for (int unit = blockIdx.x * KS_WARPS + w; unit < n_units; unit += gridDim.x * KS_WARPS) {
        uint8_t *dst = wy + (size_t)unit * kKdaUnitBytes;
        const float4 *Ag = reinterpret_cast<const float4 *>(dst);
#pragma unroll 4
        for (int e = lane; e < C * C / 4; e += 32) {
            const int i = e / (C / 4), j = 4 * (e % (C / 4));
            *reinterpret_cast<float4 *>(S + i * kLS + j) = Ag[e];
        }
        const float *bg = reinterpret_cast<const float *>(dst + 2 * kWyTileBytes);
        beta[lane] = bg[lane];
        beta[32 + lane] = bg[32 + lane];
        __syncwarp();
        solve_unit(S, dst, beta, one);
        __syncwarp();
    }
}

}  // namespace

int launch_tc_kda_prep(const cpdr_ctx *c, const void *k, const void *q, const void *beta, const float *g,
                       void *wy, void *stream) {
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
    prm.H = pl.H;
    cudaError_t e = cudaFuncSetAttribute(tc_kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)KP_SMEM);
    if (e != cudaSuccess) return (int)e;
    tc_kda_prep_kernel<<<(unsigned)units, KP_THREADS, KP_SMEM, (cudaStream_t)stream>>>(prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    const size_t ssm = KS_WARPS * KS_SCRATCH;
    e = cudaFuncSetAttribute(tc_kda_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return (int)e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int64_t blocks = (units + KS_WARPS - 1) / KS_WARPS;
    const int grid = (int)std::min<int64_t>(blocks, (int64_t)sms * 3);
    tc_kda_solve_kernel<<<grid, 32 * KS_WARPS, ssm, (cudaStream_t)stream>>>((uint8_t *)wy, (int)units);
    return (int)cudaGetLastError();
}

}  // namespace cpdr
