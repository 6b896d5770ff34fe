// WY build on the tensor-core path (bf16, d = 128, scalar gate): for every
// 64-token chunk of every fragment and every head ([FLA-CP] §2.2, the
// recompute_w_u step of its §4 Code Flow)
//   P  = K K^T                                          (tcgen05, fp32 in TMEM)
//   A  = beta_i 2^(G_i - G_j) P_ij, j < i               (SIMT)
//   T  = (I + A)^-1                                     (SIMT, fp32)
//   T' = T diag(beta),  T'' = T diag(beta gamma),  gamma_j = 2^(G_j)
// written as three bf16 64 x 64 tiles per (chunk, head) "unit": T', hi(T'')
// and lo(T'') = bf16(T'' - hi(T'')), each the 8 KiB 128-byte-swizzled image
// the chain kernels' MMAs read (K-major rows i, columns j).
//
// The solves of different chunks are independent, so they run here in one
// fully parallel launch; the chain kernels (tc_chain.cu) stream the tiles.
//
// CTA = 17 warps, 8 units per iteration.  Warp 16 issues the loads and MMAs:
// one M = 128, N = 128 MMA per pair of units computes [K_a; K_b][K_a; K_b]^T,
// whose diagonal blocks are K_a K_a^T (TMEM lanes 0..63) and K_b K_b^T (lanes
// 64..127); four pairs fill the 512 TMEM columns.  Warps 0..15 first form A
// for every unit from TMEM (warp w: 32 rows of pair w / 4 from its own TMEM
// lane quarter w % 4), then warps 2u and 2u + 1 solve unit u together by
// 32 x 32 blocks (tc_solve.cuh): each inverts one diagonal block by forward
// substitution, T_i = e_i - sum_{k<i} A_ik T_k, with its column in registers,
// then the two share the off-diagonal block's products by rows.  The pair
// halves the serial depth of a solve and puts four solver warps on each SM
// sub-partition.  The next iteration's K tiles and products are issued while
// the units are being solved.  Waits are bounded as in the chain kernels.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"
#include "tc_gates.cuh"
#include "tc_solve.cuh"

namespace cpdr {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int WY_SOLVERS = 8;                     // units per iteration
constexpr int WY_WARPS = 2 * WY_SOLVERS;          // solver warps: a pair per unit
constexpr int WY_THREADS = 32 * (WY_WARPS + 1);
constexpr uint32_t WY_TMEM_COLS = 512;

// Shared-memory carve-up (byte offsets from a 1024-aligned base)
constexpr uint32_t O_KT = 0;                      // 2 pair buffers [a.c0 | b.c0 | a.c1 | b.c1], 32 KiB each
constexpr uint32_t O_SCR = 65536;                 // 8 units x [64][68] fp32
constexpr uint32_t SCR_BYTES = 64 * kLS * 4;
constexpr int kWyGateFloats = 5 * 64 + 4;         // G, beta, gamma, e, f, flag
constexpr uint32_t O_GATES = O_SCR + WY_SOLVERS * SCR_BYTES;   // 2 slots x 8 units
constexpr uint32_t O_BARS = O_GATES + 2 * WY_SOLVERS * kWyGateFloats * 4;
enum WyBar { WB_KFULL0, WB_KFULL1, WB_KFREE0, WB_KFREE1, WB_PFULL, WB_TFREE, WB_DRAIN, WB_N };
constexpr uint32_t O_CTL = O_BARS + 64;
constexpr uint32_t O_TSLOT = O_CTL + 16;
constexpr uint32_t WY_SMEM = O_TSLOT + 16;
static_assert(WY_SMEM + 1024 <= 232448, "WY layout exceeds shared memory");
constexpr int kSolveBarId = 1;                    // named barrier of the 16 solver warps
constexpr int kPairBarId0 = 2;                    // named barriers 2 .. 9: one per solver pair

struct WyParams {
    const WyChunk *chunks;
    const __nv_bfloat16 *beta;
    const float *g;
    uint8_t *wy;
    float *tmat;   // nullable: T of every unit as fp32 64 x 64 (the backward's input gradients read it)
    int32_t *status;
    int n_units;   // chunks x heads
    int H;
};

struct WyGates {
    float *G, *beta, *gam, *e, *f, *flag;
};
__device__ __forceinline__ WyGates wy_gates(uint8_t *base, int slot, int unit) {
    float *q = reinterpret_cast<float *>(base + O_GATES) + (slot * WY_SOLVERS + unit) * kWyGateFloats;
    return WyGates{q, q + 64, q + 128, q + 192, q + 256, q + 320};
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool wy_warp_wait(uint64_t *bar, uint32_t parity, Ctl *ctl, int32_t *status, int site) {
    return warp_wait_all(bar, parity, ctl, status, site);
}

// beta and log2 gates of rows 2*lane, 2*lane+1 of a unit (padded rows: 0)
struct GateIn {
    float b0, b1, g0, g1;
};
__device__ __forceinline__ GateIn load_gate_inputs(const WyParams &p, int unit) {
    GateIn r{0.f, 0.f, 0.f, 0.f};
    if (unit >= p.n_units) return r;
    const int lane = threadIdx.x & 31;
    const WyChunk ck = p.chunks[unit / p.H];
    const int h = unit % p.H;
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    if (i0 < ck.nv) {
        r.b0 = __bfloat162float(p.beta[(ck.tok0 + i0) * p.H + h]);
        r.g0 = p.g[(ck.tok0 + i0) * p.H + h] * kLog2e;
    }
    if (i1 < ck.nv) {
        r.b1 = __bfloat162float(p.beta[(ck.tok0 + i1) * p.H + h]);
        r.g1 = p.g[(ck.tok0 + i1) * p.H + h] * kLog2e;
    }
    return r;
}
__device__ __forceinline__ void write_gates(const WyGates &gs, const GateIn &in) {
    const int lane = threadIdx.x & 31;
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    const LaneGates lg = scan_gates(in.g0, in.g1);
    gs.G[i0] = lg.G0; gs.G[i1] = lg.G1;
    gs.beta[i0] = in.b0; gs.beta[i1] = in.b1;
    gs.gam[i0] = exp2f(lg.G0); gs.gam[i1] = exp2f(lg.G1);
    gs.e[i0] = exp2f(lg.G0 - lg.Gr); gs.e[i1] = exp2f(lg.G1 - lg.Gr);
    gs.f[i0] = exp2f(lg.Gr - lg.G0); gs.f[i1] = exp2f(lg.Gr - lg.G1);
    if (lane == 0) gs.flag[0] = lg.exact ? 1.f : 0.f;
}

__global__ void __launch_bounds__(WY_THREADS, 1)
tc_wy_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ WyParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + O_BARS);
    Ctl *ctl = reinterpret_cast<Ctl *>(base + O_CTL);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + O_TSLOT);
    const int ngroups = (p.n_units + WY_SOLVERS - 1) / WY_SOLVERS;
    const int H = p.H;

    if (tid == 0) {
        mbar_init(&bar[WB_KFULL0], 1);
        mbar_init(&bar[WB_KFULL1], 1);
        mbar_init(&bar[WB_KFREE0], 1);
        mbar_init(&bar[WB_KFREE1], 1);
        mbar_init(&bar[WB_PFULL], 1);
        mbar_init(&bar[WB_TFREE], WY_WARPS);
        mbar_init(&bar[WB_DRAIN], 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == WY_WARPS) {
        if (lane == 0) tma_prefetch_desc(&tk);
        tmem_alloc(tslot, WY_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (w == WY_WARPS) {
        // ---------------------------------------------------------- loads and products
        if (lane == 0) {
            const uint32_t b0 = smem_u32(base);
            int nload[2] = {0, 0}, nmma[2] = {0, 0};
            int it = 0;
            for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x, it++) {
                bool ok = true;
                for (int hp = 0; hp < 2 && ok; hp++) {
                    // pairs 2hp and 2hp + 1 into buffers 0 and 1 (units past the
                    // end load a valid tile; their products are not used)
                    for (int b = 0; b < 2 && ok; b++) {
                        if (nload[b] > 0 && !mbar_wait(&bar[WB_KFREE0 + b], (nload[b] - 1) & 1, ctl, p.status, 84)) {
                            ok = false;
                            break;
                        }
                        const int pair = 2 * hp + b;
                        uint8_t *kt = base + O_KT + b * 32768;
                        mbar_arrive_expect_tx(&bar[WB_KFULL0 + b], 32768u);
                        for (int s = 0; s < 2; s++) {
                            int u = grp * WY_SOLVERS + 2 * pair + s;
                            if (u >= p.n_units) u = 0;
                            const int h = u % H, tok = (int)p.chunks[u / H].tok0;
                            tma_load_3d(kt + 8192 * s, &tk, &bar[WB_KFULL0 + b], 0, h, tok);
                            tma_load_3d(kt + 16384 + 8192 * s, &tk, &bar[WB_KFULL0 + b], 64, h, tok);
                        }
                        nload[b]++;
                    }
                    if (!ok) break;
                    // TMEM is free once the previous iteration's A rows were read
                    if (hp == 0 && it > 0 && !mbar_wait(&bar[WB_TFREE], (it - 1) & 1, ctl, p.status, 85)) {
                        ok = false;
                        break;
                    }
                    for (int b = 0; b < 2; b++) {
                        if (!mbar_wait(&bar[WB_KFULL0 + b], (nload[b] - 1) & 1, ctl, p.status, 86)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t d_kt = sdesc(b0 + O_KT + b * 32768, 16, 1024);
                        const uint32_t dcol = tmem + 128u * (uint32_t)(2 * hp + b);
#pragma unroll
                        for (int k = 0; k < D / 16; k++) {
                            const uint64_t o = (uint64_t)(((k & 3) * 32 + (k >> 2) * 16384) >> 4);
                            mma_bf16(dcol, d_kt + o, d_kt + o, idesc_bf16(128, 128, false, false), k > 0 ? 1u : 0u);
                        }
                        mma_commit(&bar[WB_KFREE0 + b]);
                        nmma[b]++;
                    }
                }
                if (!ok) break;
                mma_commit(&bar[WB_PFULL]);
            }
            // drain: every load consumed or landed, every product complete
            Ctl local;
            local.abort = 0;
            for (int b = 0; b < 2; b++)
                if (nload[b] > nmma[b]) mbar_wait(&bar[WB_KFULL0 + b], (nload[b] - 1) & 1, &local, p.status, 87);
            mma_commit(&bar[WB_DRAIN]);
            mbar_wait(&bar[WB_DRAIN], 0, &local, p.status, 88);
        }
    } else {
        // ---------------------------------------------------------- form and solve
        const int q = w & 3, pair = w >> 2;
        const int u_own = w >> 1, role = w & 1;   // the unit this warp solves, and its part
        // gates of this pair's first unit
        if ((int)blockIdx.x < ngroups && role == 0) {
            const int u0 = blockIdx.x * WY_SOLVERS + u_own;
            if (u0 < p.n_units) write_gates(wy_gates(base, 0, u_own), load_gate_inputs(p, u0));
        }
        named_bar(kSolveBarId, 32 * WY_WARPS);
        int it = 0;
        for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x, it++) {
            const int slot = it & 1;
            const bool pok = wy_warp_wait(&bar[WB_PFULL], it & 1, ctl, p.status, 89);
            if (pok) {
                tc_fence_after();
                // A rows from TMEM: lanes 32q.. of pair w / 4; unit a of the
                // pair (q < 2) holds lanes 0..63, unit b (q >= 2) 64..127
                const int ul = 2 * pair + (q >> 1);
                if (grp * WY_SOLVERS + ul < p.n_units) {
                    const WyGates gs = wy_gates(base, slot, ul);
                    float *S = reinterpret_cast<float *>(base + O_SCR + ul * SCR_BYTES);
                    const int i = 32 * (q & 1) + lane;
                    const bool exact = gs.flag[0] != 0.f;
                    const float bi = gs.beta[i], Gi = gs.G[i], bei = gs.beta[i] * gs.e[i];
#pragma unroll
                    for (int half = 0; half < 2; half++) {
                        float vv[32];
                        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 128u * pair + 64u * (q >> 1) + 32u * half, vv);
                        tmem_ld_wait();
#pragma unroll
                        for (int q4 = 0; q4 < 8; q4++) {
                            const int j0 = 32 * half + 4 * q4;
                            const float4 f4 = *reinterpret_cast<const float4 *>(gs.f + j0);
                            const float fv[4] = {f4.x, f4.y, f4.z, f4.w};
                            float e4[4];
                            if (exact) {   // steep gates: the factored form could overflow
#pragma unroll
                                for (int u = 0; u < 4; u++)
                                    e4[u] = (j0 + u < i) ? bi * exp2f(Gi - gs.G[j0 + u]) * vv[4 * q4 + u] : 0.f;
                            } else {
#pragma unroll
                                for (int u = 0; u < 4; u++)
                                    e4[u] = (j0 + u < i) ? bei * fv[u] * vv[4 * q4 + u] : 0.f;
                            }
                            *reinterpret_cast<float4 *>(S + i * kLS + j0) = make_float4(e4[0], e4[1], e4[2], e4[3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[WB_TFREE]);
            }
            // every unit's A is in place; leave together if any wait gave up
            if (named_bar_or(kSolveBarId, 32 * WY_WARPS, pok ? 0 : 1)) break;
            const int unit = grp * WY_SOLVERS + u_own;
            // the next iteration's gate inputs load while this unit is solved
            const int ngrp = grp + gridDim.x;
            const bool nxt_ok = role == 0 && ngrp < ngroups && ngrp * WY_SOLVERS + u_own < p.n_units;
            const GateIn nxt = load_gate_inputs(p, nxt_ok ? ngrp * WY_SOLVERS + u_own : p.n_units);
            if (unit < p.n_units) {
                float *S = reinterpret_cast<float *>(base + O_SCR + u_own * SCR_BYTES);
                const WyGates gs = wy_gates(base, slot, u_own);
                solve_unit_pair(S, p.wy + (size_t)unit * kWyUnitBytes, gs.beta, gs.gam, role, kPairBarId0 + u_own,
                                p.tmat ? p.tmat + (size_t)unit * 64 * 64 : nullptr);
            }
            if (nxt_ok) write_gates(wy_gates(base, slot ^ 1, u_own), nxt);
            named_bar(kSolveBarId, 32 * WY_WARPS);   // scratch and gate slot free
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == WY_WARPS) tmem_dealloc(tmem, WY_TMEM_COLS);
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
    const size_t units = c->plan.wy_chunks.size() * (size_t)c->plan.H;
    if (c->plan.gate_kind != CPDR_GATE_PER_DIM) return units * kWyUnitBytes;
    return units * (kKdaUnitBytes + (size_t)(c->plan.G - 1) * kKdaQpBytes);
}

int launch_tc_wy(const cpdr_ctx *c, const void *k, const void *beta, const float *g, void *wy, void *stream) {
    return launch_tc_wy_t(c, k, beta, g, wy, nullptr, stream);
}

int launch_tc_wy_t(const cpdr_ctx *c, const void *k, const void *beta, const float *g, void *wy, float *tmat,
                   void *stream) {
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
    prm.tmat = tmat;
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
    const int ngroups = (int)((units + WY_SOLVERS - 1) / WY_SOLVERS);
    const int grid = ngroups < sms ? ngroups : sms;
    tc_wy_kernel<<<grid, WY_THREADS, smem, (cudaStream_t)stream>>>(tk, prm);
    return (int)cudaGetLastError();
}

}  // namespace cpdr
