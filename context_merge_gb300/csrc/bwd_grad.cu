// Input gradients of the chunked backward, one CTA per (chunk, head) unit,
// all units in parallel (bf16 inputs, d = 128, scalar gate).  With grouped
// query heads the unit makes one pass per query head of its state for dq
// and the q, dO parts of dk and dG (dS' and dDelta already sum over them).
//
// The chunk form of the article "flash-linear-attention 上下文并行CP ..."
// ([FLA-CP] §2.2; the backward flow of §4) gives, per chunk, with the state
// S at the chunk's start, Delta = U - W S, the state gradient dS' after the
// chunk and dDelta (the last two from the state-gradient chain, tc_chain.cu
// MODE_BWD), dO~ = scale dO, in-chunk log gates G_i (natural log), gamma_i =
// e^G_i, Gamma_i = e^(G_C - G_i), Lambda_ij = e^(G_i - G_j) (j <= i), and
// T = (I + A)^-1 with A_ij = beta_i Y_ij (j < i), Y = (K K^T) ⊙ Lambda:
//   dP   = lower_incl(dO~ Delta^T);  dPL = dP ⊙ Lambda
//   dq   = gamma ⊙ (dO~ S^T) + dPL K
//   dW   = -dDelta S^T;  TtW = T^T dW;  TtU = T^T dDelta
//   dv   = beta ⊙ TtU
//   W    = T diag(beta gamma) K,  U = T diag(beta) V
//   dA   = -strict_lower(TtW W^T + TtU U^T);  dAL = diag(beta) dA ⊙ Lambda
//   dk   = gamma ⊙ beta ⊙ TtW + dAL K            (through K gamma)
//        + dPL^T Q + dAL^T K                    (through K / gamma)
//        + Gamma ⊙ (Delta dS'^T)                (through Gamma ⊙ K)
//   dbeta_i = sum_d (TtW ⊙ K gamma + TtU ⊙ V)_id + sum_j dA_ij Y_ij
//   dG_i = sum_d [q ⊙ dq + k ⊙ (dk_gamma - dk_1/gamma - dk_Gamma)]_id,
//   dG_C += sum_id (k ⊙ dk_Gamma)_id + gamma^C sum_d (dS' ⊙ S)_dd'  (summed)
//   dg_t = sum_{s >= t in the chunk} dG_s
// — the reverse-mode derivative of the chunk equations, written with every
// gate factor as a bounded e^(G_i - G_j), j <= i.  The matrix products run
// on the tensor cores as warp-level mma.sync (tf32 operands, fp32
// accumulation) from shared memory; T comes from the WY build (fp32).  Rows
// past the chunk's end are zero and not written.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "bwd_mma.cuh"

namespace cpdr {
namespace {

using namespace bwdmm;

constexpr int D = 128;
constexpr int C = 64;
constexpr int NT = 256;          // 8 warps
constexpr int PB = D + 8;        // bf16 row pitch (elements)
constexpr int PF = D + 4;        // fp32 row pitch of 64 x 128 / 128 x 128 tiles
constexpr int PS = C + 4;        // fp32 row pitch of 64 x 64 tiles

struct GradParams {
    const WyChunk *chunks;       // per global chunk: first token, valid rows
    const __nv_bfloat16 *q, *k, *v, *beta, *dout;
    const float *g;
    const float *T;                  // per unit: the WY inverse T = (I + A)^-1, 64 x 64 (from the WY build)
    const float *S, *Dl, *dS, *dD;   // per unit: S [dk][dv], Delta [64][dv], dS' [dk][dv], dDelta [64][dv]
    float *dq, *dk, *dv, *dbeta, *dg;
    int H, G;                        // state heads; query heads per state (q, dO, dq have G H heads)
    float scale;
};

// shared memory (bytes)
constexpr int OFF_QB = 0;
constexpr int OFF_KB = OFF_QB + C * PB * 2;
constexpr int OFF_VB = OFF_KB + C * PB * 2;
constexpr int OFF_OB = OFF_VB + C * PB * 2;
constexpr int OFF_DL = OFF_OB + C * PB * 2;          // Delta, then TtU
constexpr int OFF_DD = OFF_DL + C * PF * 4;          // dDelta, then U
constexpr int OFF_R = OFF_DD + C * PF * 4;           // S / dS' halves, then W
constexpr int OFF_W = OFF_R + C * PF * 4;            // dW, then TtW
// 64 x 64 fp32 tiles: T1 = dPL, then Y, in dO's rows once dO is dead (a warp
// writes only the rows it read; the row pitches match); T2 = T, then dAL
constexpr int OFF_T1 = OFF_OB;
constexpr int OFF_T2 = OFF_W + C * PF * 4;
constexpr int OFF_T3 = OFF_T2;
constexpr int OFF_VEC = OFF_T2 + C * PS * 4;         // G, gam, Gam, beta, dG, dbeta (64 each), misc, solve sums
constexpr int SMEM = OFF_VEC + (6 * C + 16) * 4;
static_assert(PS * 4 == PB * 2, "T1 rows must overlay dO rows");
static_assert(SMEM <= 232448, "gradient kernel shared memory");

// GQA: several query heads per state (a pass per query head); without it
// the single pass compiles with its branches resolved.
template <bool GQA>
__global__ void __launch_bounds__(NT, 1) bwd_grad_kernel(const __grid_constant__ GradParams p) {
    extern __shared__ __align__(16) uint8_t sm[];
    __nv_bfloat16 *Qb = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_QB);
    __nv_bfloat16 *Kb = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_KB);
    __nv_bfloat16 *Vb = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_VB);
    __nv_bfloat16 *Ob = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_OB);
    float *DL = reinterpret_cast<float *>(sm + OFF_DL);
    float *DD = reinterpret_cast<float *>(sm + OFF_DD);
    float *R = reinterpret_cast<float *>(sm + OFF_R);
    float *WB = reinterpret_cast<float *>(sm + OFF_W);
    float *T1 = reinterpret_cast<float *>(sm + OFF_T1);
    float *T2 = reinterpret_cast<float *>(sm + OFF_T2);
    float *T3 = reinterpret_cast<float *>(sm + OFF_T3);
    float *Gv = reinterpret_cast<float *>(sm + OFF_VEC);
    float *gam = Gv + C, *Gam = Gv + 2 * C, *bet = Gv + 3 * C, *dGrow = Gv + 4 * C, *dbet = Gv + 5 * C;
    float *misc = Gv + 6 * C;   // [0] gamma^C, [1] dG_C accumulator

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, tg = lane & 3;
    const int64_t unit = blockIdx.x;
    const int h = (int)(unit % p.H);
    const WyChunk ck = p.chunks[unit / p.H];
    const int nv = ck.nv;
    auto tok = [&](int i) { return (ck.tok0 + i) * p.H + h; };
    // row i of query head gq of this state
    auto qtok = [&](int i, int gq) { return ((ck.tok0 + i) * p.H + h) * p.G + gq; };

    // q and dO of query head gq into Qb, Ob (rows past the chunk's end: 0)
    auto load_qo = [&](int gq) {
        for (int e = tid; e < C * (D / 8); e += NT) {
            const int i = e / (D / 8), d = 8 * (e % (D / 8));
            uint4 qv = make_uint4(0, 0, 0, 0), ov = qv;
            if (i < nv) {
                const int64_t o = (int64_t)qtok(i, gq) * D + d;
                qv = *reinterpret_cast<const uint4 *>(p.q + o);
                ov = *reinterpret_cast<const uint4 *>(p.dout + o);
            }
            *reinterpret_cast<uint4 *>(Qb + i * PB + d) = qv;
            *reinterpret_cast<uint4 *>(Ob + i * PB + d) = ov;
        }
    };
    // ---- loads (rows past the chunk's end: 0): q, dO of the first query
    // head, k, v (one loop: every load independent), then Delta, dDelta
    for (int e = tid; e < C * (D / 8); e += NT) {
        const int i = e / (D / 8), d = 8 * (e % (D / 8));
        uint4 qv = make_uint4(0, 0, 0, 0), kv = qv, vv = qv, ov = qv;
        if (i < nv) {
            const int64_t o = (int64_t)tok(i) * D + d, oq = (int64_t)qtok(i, 0) * D + d;
            qv = *reinterpret_cast<const uint4 *>(p.q + oq);
            kv = *reinterpret_cast<const uint4 *>(p.k + o);
            vv = *reinterpret_cast<const uint4 *>(p.v + o);
            ov = *reinterpret_cast<const uint4 *>(p.dout + oq);
        }
        *reinterpret_cast<uint4 *>(Qb + i * PB + d) = qv;
        *reinterpret_cast<uint4 *>(Kb + i * PB + d) = kv;
        *reinterpret_cast<uint4 *>(Vb + i * PB + d) = vv;
        *reinterpret_cast<uint4 *>(Ob + i * PB + d) = ov;
    }
    const float *Sg = p.S + unit * D * D, *dSg = p.dS + unit * D * D;
    const float *Dlg = p.Dl + unit * C * D, *dDg = p.dD + unit * C * D;
    for (int e = tid; e < C * (D / 4); e += NT) {
        const int i = e / (D / 4), d = 4 * (e % (D / 4));
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (i < nv) {
            a = *reinterpret_cast<const float4 *>(Dlg + i * D + d);
            b = *reinterpret_cast<const float4 *>(dDg + i * D + d);
        }
        *reinterpret_cast<float4 *>(DL + i * PF + d) = a;
        *reinterpret_cast<float4 *>(DD + i * PF + d) = b;
        // the first half of dS' (the first pass starts with it) and T
        *reinterpret_cast<float4 *>(R + i * PF + d) = *reinterpret_cast<const float4 *>(dSg + (int64_t)i * D + d);
    }
    {   // T = (I + A)^-1 of this unit, solved by the WY build (fp32)
        const float *Tg = p.T + unit * C * C;
        for (int e = tid; e < C * C / 4; e += NT) {
            const int i = e / (C / 4), j = 4 * (e % (C / 4));
            *reinterpret_cast<float4 *>(T2 + i * PS + j) = *reinterpret_cast<const float4 *>(Tg + i * C + j);
        }
    }
    if (tid < C) {
        dGrow[tid] = 0.f;
        dbet[tid] = 0.f;
    }
    if (tid == 0) misc[1] = 0.f;
    // in-chunk log gates (natural log, padded rows 0)
    if (w == 0) {
        const int i0 = 2 * lane, i1 = i0 + 1;
        const float g0 = i0 < nv ? p.g[tok(i0)] : 0.f, g1 = i1 < nv ? p.g[tok(i1)] : 0.f;
        float x = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const float G1 = x, G0 = x - g1, GC = __shfl_sync(0xffffffffu, x, 31);
        Gv[i0] = G0; Gv[i1] = G1;
        gam[i0] = __expf(G0); gam[i1] = __expf(G1);
        Gam[i0] = __expf(GC - G0); Gam[i1] = __expf(GC - G1);
        bet[i0] = i0 < nv ? bf(p.beta + tok(i0)) : 0.f;
        bet[i1] = i1 < nv ? bf(p.beta + tok(i1)) : 0.f;
        if (lane == 0) misc[0] = __expf(GC);
    }

    // Register tiles of 64 x 128 outputs: warp w owns rows m0 = 16 (w % 4)
    // .. + 15 and, in each 64-column half hh, columns 64 hh + 32 (w / 4) ..
    // + 31 (four 8-column tiles); thread: rows m0 + g, m0 + g + 8, columns
    // 2 tg, 2 tg + 1 of each tile.
    const int m0 = 16 * (w & 3), cw = 32 * (w >> 2);
    const int r0 = m0 + g, r1 = m0 + g + 8;
    int n8[8], nh[2][4];
#pragma unroll
    for (int hh = 0; hh < 2; hh++)
#pragma unroll
        for (int nt = 0; nt < 4; nt++) {
            nh[hh][nt] = 64 * hh + cw + 8 * nt;
            n8[4 * hh + nt] = nh[hh][nt];
        }
    float dQ[8][4], dK[8][4];
    zero(dK);
    float dg0 = 0.f, dg1 = 0.f;   // this thread's share of dG for rows r0, r1
    float db0 = 0.f, db1 = 0.f;   // and of dbeta
    const Bv Ov{Ob, PB, 1}, Kv{Kb, PB, 1}, Qv{Qb, PB, 1};
    const Bv KvT{Kb, 1, PB};
    const float sc = p.scale;
    float dgc_part = 0.f;   // sum (dS' ⊙ S)
    float dgc_k = 0.f;      // sum (k ⊙ dk_Gamma)

    // ---- one pass per query head of this state (one without grouped query
    // heads): its dq, and its parts of dk and dG; the first pass also forms
    // dW = -dDelta S^T and sum (dS' ⊙ S) from the same S halves
    const int npass = GQA ? p.G : 1;
#pragma unroll 1
    for (int gq = 0; gq < npass; gq++) {
        const bool first = !GQA || gq == 0;
        if (!first) {
            __syncthreads();   // the previous pass's reads of Q and dO (T1) are done
            load_qo(gq);
        }
        // ---- S halves: dq_1 = gamma ⊙ (dO~ S^T) (first pass: dW = -dDelta S^T);
        // dS' halves (first pass): dk_Gamma = Gamma ⊙ (Delta dS'^T); and
        // sum (dS' ⊙ S).  One 64 x 128 fp32 half at a time in R.
        const int nl[4] = {cw, cw + 8, cw + 16, cw + 24};
        const Fv RT{R, 1, PF};   // B(v, d') = R[d'][v]
        auto s_phase = [&](int hh) {
            float acc[4][4];
            zero(acc);
            warp_mm<4, D>(acc, Ov, m0, RT, nl);
#pragma unroll
            for (int nt = 0; nt < 4; nt++) {
                dQ[4 * hh + nt][0] = sc * acc[nt][0] * gam[r0];
                dQ[4 * hh + nt][1] = sc * acc[nt][1] * gam[r0];
                dQ[4 * hh + nt][2] = sc * acc[nt][2] * gam[r1];
                dQ[4 * hh + nt][3] = sc * acc[nt][3] * gam[r1];
            }
            if (first) {
                zero(acc);
                warp_mm<4, D>(acc, Fv{DD, PF, 1}, m0, RT, nl);
#pragma unroll
                for (int nt = 0; nt < 4; nt++) {
                    const int col = 64 * hh + cw + 8 * nt + 2 * tg;
                    WB[r0 * PF + col] = -acc[nt][0];
                    WB[r0 * PF + col + 1] = -acc[nt][1];
                    WB[r1 * PF + col] = -acc[nt][2];
                    WB[r1 * PF + col + 1] = -acc[nt][3];
                }
            }
        };
        auto ds_phase = [&](int hh) {
            float acc[4][4];
            zero(acc);
            warp_mm<4, D>(acc, Fv{DL, PF, 1}, m0, RT, nl);
#pragma unroll
            for (int nt = 0; nt < 4; nt++) {
                const int col = 64 * hh + cw + 8 * nt + 2 * tg;
                const float v0 = Gam[r0] * acc[nt][0], v1 = Gam[r0] * acc[nt][1];
                const float v2 = Gam[r1] * acc[nt][2], v3 = Gam[r1] * acc[nt][3];
                dK[4 * hh + nt][0] += v0; dK[4 * hh + nt][1] += v1;
                dK[4 * hh + nt][2] += v2; dK[4 * hh + nt][3] += v3;
                const float k0 = bf(Kb + r0 * PB + col) * v0 + bf(Kb + r0 * PB + col + 1) * v1;
                const float k1 = bf(Kb + r1 * PB + col) * v2 + bf(Kb + r1 * PB + col + 1) * v3;
                dg0 -= k0;
                dg1 -= k1;
                dgc_k += k0 + k1;
            }
        };
        if (first) {
            // the next half's global loads are in flight (registers: a thread
            // holds rows w + 8 m, columns 4 lane) while the current half is used;
            // R starts with dS' half 0 (loaded with the inputs)
            float4 pf[8];
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const float *sh = Sg + (int64_t)64 * hh * D;   // S half hh in flight
#pragma unroll
                for (int m = 0; m < 8; m++) pf[m] = *reinterpret_cast<const float4 *>(sh + (w + 8 * m) * D + 4 * lane);
                __syncthreads();
                ds_phase(hh);
#pragma unroll
                for (int m = 0; m < 8; m++) {   // sum (dS' ⊙ S) over this thread's elements
                    const float4 x = *reinterpret_cast<const float4 *>(R + (w + 8 * m) * PF + 4 * lane);
                    dgc_part += x.x * pf[m].x + x.y * pf[m].y + x.z * pf[m].z + x.w * pf[m].w;
                }
                __syncthreads();
#pragma unroll
                for (int m = 0; m < 8; m++) *reinterpret_cast<float4 *>(R + (w + 8 * m) * PF + 4 * lane) = pf[m];
                if (hh == 0) {   // dS' half 1 in flight
#pragma unroll
                    for (int m = 0; m < 8; m++)
                        pf[m] = *reinterpret_cast<const float4 *>(dSg + (64 + w + 8 * m) * D + 4 * lane);
                }
                __syncthreads();
                s_phase(hh);
                if (hh == 0) {
                    __syncthreads();
#pragma unroll
                    for (int m = 0; m < 8; m++) *reinterpret_cast<float4 *>(R + (w + 8 * m) * PF + 4 * lane) = pf[m];
                }
            }
        } else {
            for (int hh = 0; hh < 2; hh++) {
                __syncthreads();
                for (int e = tid; e < C * (D / 4); e += NT) {
                    const int i = e / (D / 4), d = 4 * (e % (D / 4));
                    *reinterpret_cast<float4 *>(R + i * PF + d) =
                        *reinterpret_cast<const float4 *>(Sg + (int64_t)(64 * hh + i) * D + d);
                }
                __syncthreads();
                s_phase(hh);
            }
        }
        __syncthreads();
        // ---- dP = lower_incl(dO~ Delta^T), dPL = dP ⊙ Lambda  (64 x 64 into T1)
        {
            const int nl[4] = {cw, cw + 8, cw + 16, cw + 24};
            float acc[4][4];
            zero(acc);
            warp_mm<4, D>(acc, Ov, m0, Fv{DL, 1, PF}, nl);
            __syncthreads();   // T1 overlays dO: the other column warp reads these rows
#pragma unroll
            for (int nt = 0; nt < 4; nt++) {
                const int j = cw + 8 * nt + 2 * tg;
                auto lam = [&](int i, int jj) { return jj <= i ? __expf(Gv[i] - Gv[jj]) : 0.f; };
                T1[r0 * PS + j] = sc * acc[nt][0] * lam(r0, j);
                T1[r0 * PS + j + 1] = sc * acc[nt][1] * lam(r0, j + 1);
                T1[r1 * PS + j] = sc * acc[nt][2] * lam(r1, j);
                T1[r1 * PS + j + 1] = sc * acc[nt][3] * lam(r1, j + 1);
            }
        }
        __syncthreads();
        // dq += dPL K;  dk_1 = dPL^T Q (through K / gamma)
        {
            warp_mm<8, C>(dQ, Fv{T1, PS, 1}, m0, Kv, n8);
            float acc[8][4];
            zero(acc);
            warp_mm<8, C>(acc, Fv{T1, 1, PS}, m0, Qv, n8);
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                const int col = n8[nt] + 2 * tg;
#pragma unroll
                for (int e = 0; e < 4; e++) dK[nt][e] += acc[nt][e];
                dg0 -= bf(Kb + r0 * PB + col) * acc[nt][0] + bf(Kb + r0 * PB + col + 1) * acc[nt][1];
                dg1 -= bf(Kb + r1 * PB + col) * acc[nt][2] + bf(Kb + r1 * PB + col + 1) * acc[nt][3];
            }
        }
        // ---- dq of this query head; dG_i += sum_d q dq
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            dg0 += bf(Qb + r0 * PB + col) * dQ[nt][0] + bf(Qb + r0 * PB + col + 1) * dQ[nt][1];
            dg1 += bf(Qb + r1 * PB + col) * dQ[nt][2] + bf(Qb + r1 * PB + col + 1) * dQ[nt][3];
            if (r0 < nv)
                *reinterpret_cast<float2 *>(p.dq + (int64_t)qtok(r0, gq) * D + col) = make_float2(dQ[nt][0], dQ[nt][1]);
            if (r1 < nv)
                *reinterpret_cast<float2 *>(p.dq + (int64_t)qtok(r1, gq) * D + col) = make_float2(dQ[nt][2], dQ[nt][3]);
        }
    }
    __syncthreads();
    // ---- Y = (K K^T) ⊙ Lambda into T1 (lower incl.); A = beta_i Y_ij (j < i)
    {
        const int nl[4] = {cw, cw + 8, cw + 16, cw + 24};
        float acc[4][4];
        zero(acc);
        warp_mm<4, D>(acc, Kv, m0, KvT, nl);
#pragma unroll
        for (int nt = 0; nt < 4; nt++) {
            const int j = cw + 8 * nt + 2 * tg;
            auto lam = [&](int i, int jj) { return jj <= i ? __expf(Gv[i] - Gv[jj]) : 0.f; };
            T1[r0 * PS + j] = acc[nt][0] * lam(r0, j);
            T1[r0 * PS + j + 1] = acc[nt][1] * lam(r0, j + 1);
            T1[r1 * PS + j] = acc[nt][2] * lam(r1, j);
            T1[r1 * PS + j + 1] = acc[nt][3] * lam(r1, j + 1);
        }
    }
    __syncthreads();
    __syncthreads();
    // ---- TtW = T^T dW, TtU = T^T dDelta (64 x 128, register tiles); T was loaded with the inputs
    const Fv TT{T2, 1, PS};
    {
        float acc[8][4];
        zero(acc);
        warp_mm<8, C>(acc, TT, m0, Fv{WB, PF, 1}, n8);
        // dk += gamma beta TtW, dbeta += sum_d TtW K gamma, dG += k ⊙ (gamma beta TtW)
        const float gb0 = gam[r0] * bet[r0], gb1 = gam[r1] * bet[r1];
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            const float k00 = bf(Kb + r0 * PB + col), k01 = bf(Kb + r0 * PB + col + 1);
            const float k10 = bf(Kb + r1 * PB + col), k11 = bf(Kb + r1 * PB + col + 1);
            dK[nt][0] += gb0 * acc[nt][0]; dK[nt][1] += gb0 * acc[nt][1];
            dK[nt][2] += gb1 * acc[nt][2]; dK[nt][3] += gb1 * acc[nt][3];
            db0 += gam[r0] * (acc[nt][0] * k00 + acc[nt][1] * k01);
            db1 += gam[r1] * (acc[nt][2] * k10 + acc[nt][3] * k11);
            dg0 += gb0 * (acc[nt][0] * k00 + acc[nt][1] * k01);
            dg1 += gb1 * (acc[nt][2] * k10 + acc[nt][3] * k11);
        }
        __syncthreads();   // every warp has read dW
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            WB[r0 * PF + col] = acc[nt][0]; WB[r0 * PF + col + 1] = acc[nt][1];
            WB[r1 * PF + col] = acc[nt][2]; WB[r1 * PF + col + 1] = acc[nt][3];
        }
    }
    {
        float acc[8][4];
        zero(acc);
        warp_mm<8, C>(acc, TT, m0, Fv{DD, PF, 1}, n8);
        // dv = beta TtU, dbeta += sum_d TtU V
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            db0 += acc[nt][0] * bf(Vb + r0 * PB + col) + acc[nt][1] * bf(Vb + r0 * PB + col + 1);
            db1 += acc[nt][2] * bf(Vb + r1 * PB + col) + acc[nt][3] * bf(Vb + r1 * PB + col + 1);
            if (r0 < nv) {
                float2 *o = reinterpret_cast<float2 *>(p.dv + (int64_t)tok(r0) * D + col);
                *o = make_float2(bet[r0] * acc[nt][0], bet[r0] * acc[nt][1]);
            }
            if (r1 < nv) {
                float2 *o = reinterpret_cast<float2 *>(p.dv + (int64_t)tok(r1) * D + col);
                *o = make_float2(bet[r1] * acc[nt][2], bet[r1] * acc[nt][3]);
            }
        }
        __syncthreads();   // every warp has read dDelta
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            DL[r0 * PF + col] = acc[nt][0]; DL[r0 * PF + col + 1] = acc[nt][1];   // TtU replaces Delta
            DL[r1 * PF + col] = acc[nt][2]; DL[r1 * PF + col + 1] = acc[nt][3];
        }
    }
    // ---- W = T diag(beta gamma) K (into R), U = T diag(beta) V (into DD)
    {
        struct BKs {
            const __nv_bfloat16 *p;
            const float *s1, *s2;
            __device__ __forceinline__ float at(int r, int c) const { return bf(p + r * PB + c) * s1[r] * s2[r]; }
        };
        struct BVs {
            const __nv_bfloat16 *p;
            const float *s1;
            __device__ __forceinline__ float at(int r, int c) const { return bf(p + r * PB + c) * s1[r]; }
        };
        float acc[8][4];
        zero(acc);
        warp_mm<8, C>(acc, Fv{T2, PS, 1}, m0, BKs{Kb, bet, gam}, n8);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            R[r0 * PF + col] = acc[nt][0]; R[r0 * PF + col + 1] = acc[nt][1];
            R[r1 * PF + col] = acc[nt][2]; R[r1 * PF + col + 1] = acc[nt][3];
        }
        zero(acc);
        warp_mm<8, C>(acc, Fv{T2, PS, 1}, m0, BVs{Vb, bet}, n8);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
            DD[r0 * PF + col] = acc[nt][0]; DD[r0 * PF + col + 1] = acc[nt][1];
            DD[r1 * PF + col] = acc[nt][2]; DD[r1 * PF + col + 1] = acc[nt][3];
        }
    }
    __syncthreads();
    // ---- dA = -strict_lower(TtW W^T + TtU U^T); dbeta += sum_j dA Y; dAL = beta dA ⊙ Lambda (T3)
    {
        const int nl[4] = {cw, cw + 8, cw + 16, cw + 24};
        float acc[4][4];
        zero(acc);
        warp_mm<4, D>(acc, Fv{WB, PF, 1}, m0, Fv{R, 1, PF}, nl);
        warp_mm<4, D>(acc, Fv{DL, PF, 1}, m0, Fv{DD, 1, PF}, nl);
#pragma unroll
        for (int nt = 0; nt < 4; nt++) {
            const int j = cw + 8 * nt + 2 * tg;
            float a[4] = {acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]};
            const int ri[4] = {r0, r0, r1, r1}, cj[4] = {j, j + 1, j, j + 1};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int i = ri[e], jj = cj[e];
                const float dA = jj < i ? -a[e] : 0.f;
                if (e < 2) db0 += dA * T1[i * PS + jj]; else db1 += dA * T1[i * PS + jj];
                T3[i * PS + jj] = jj < i ? bet[i] * dA * __expf(Gv[i] - Gv[jj]) : 0.f;
            }
        }
    }
    __syncthreads();
    // ---- dk += dAL K (through K gamma) + dAL^T K (through K / gamma)
    {
        float acc[8][4];
        zero(acc);
        warp_mm<8, C>(acc, Fv{T3, PS, 1}, m0, Kv, n8);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
#pragma unroll
            for (int e = 0; e < 4; e++) dK[nt][e] += acc[nt][e];
            dg0 += bf(Kb + r0 * PB + col) * acc[nt][0] + bf(Kb + r0 * PB + col + 1) * acc[nt][1];
            dg1 += bf(Kb + r1 * PB + col) * acc[nt][2] + bf(Kb + r1 * PB + col + 1) * acc[nt][3];
        }
        zero(acc);
        warp_mm<8, C>(acc, Fv{T3, 1, PS}, m0, Kv, n8);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            const int col = n8[nt] + 2 * tg;
#pragma unroll
            for (int e = 0; e < 4; e++) dK[nt][e] += acc[nt][e];
            dg0 -= bf(Kb + r0 * PB + col) * acc[nt][0] + bf(Kb + r0 * PB + col + 1) * acc[nt][1];
            dg1 -= bf(Kb + r1 * PB + col) * acc[nt][2] + bf(Kb + r1 * PB + col + 1) * acc[nt][3];
        }
    }
    // ---- output dk
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
        const int col = n8[nt] + 2 * tg;
        if (r0 < nv)
            *reinterpret_cast<float2 *>(p.dk + (int64_t)tok(r0) * D + col) = make_float2(dK[nt][0], dK[nt][1]);
        if (r1 < nv)
            *reinterpret_cast<float2 *>(p.dk + (int64_t)tok(r1) * D + col) = make_float2(dK[nt][2], dK[nt][3]);
    }
    // row sums over the 4 lanes of a group, then over the two column warps
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        dg0 += __shfl_xor_sync(0xffffffffu, dg0, o);
        dg1 += __shfl_xor_sync(0xffffffffu, dg1, o);
        db0 += __shfl_xor_sync(0xffffffffu, db0, o);
        db1 += __shfl_xor_sync(0xffffffffu, db1, o);
    }
    // dG_C: sum (k ⊙ dk_Gamma) + gamma^C sum (dS' ⊙ S)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        dgc_k += __shfl_xor_sync(0xffffffffu, dgc_k, o);
        dgc_part += __shfl_xor_sync(0xffffffffu, dgc_part, o);
    }
    if (tg == 0) {
        atomicAdd(dGrow + r0, dg0);
        atomicAdd(dGrow + r1, dg1);
        atomicAdd(dbet + r0, db0);
        atomicAdd(dbet + r1, db1);
    }
    if (lane == 0) atomicAdd(misc + 1, dgc_k + misc[0] * dgc_part);
    __syncthreads();
    // dbeta; dg_t = sum_{s >= t} dG_s over the chunk's rows (dG_C on the last one)
    if (w == 0) {
        const int i0 = 2 * lane, i1 = i0 + 1;
        float x0 = i0 < nv ? dGrow[i0] + (i0 == nv - 1 ? misc[1] : 0.f) : 0.f;
        float x1 = i1 < nv ? dGrow[i1] + (i1 == nv - 1 ? misc[1] : 0.f) : 0.f;
        // reverse inclusive scan over rows 63 .. 0
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, s, o);
            if (lane + o < 32) s += y;
        }
        const float d1 = s - x0, d0 = s;   // rows i1 and i0
        if (i0 < nv) {
            p.dg[tok(i0)] = d0;
            p.dbeta[tok(i0)] = dbet[i0];
        }
        if (i1 < nv) {
            p.dg[tok(i1)] = d1;
            p.dbeta[tok(i1)] = dbet[i1];
        }
    }
}

}  // namespace

// Input gradients of every (chunk, head) unit (one CTA each), from the
// recomputed chunk states and Delta (st_S, st_D) and the state-gradient
// chain's dS' and dDelta (st_dS, st_dD).  dq, dk, dv, dbeta, dg: fp32.
int launch_bwd_grad(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta,
                    const float *g, const void *dout, const float *tmat, const float *st_S, const float *st_D,
                    const float *st_dS, const float *st_dD, float *dq, float *dk, float *dv, float *dbeta, float *dg,
                    void *stream) {
    const auto &pl = c->plan;
    const int64_t units = (int64_t)pl.wy_chunks.size() * pl.H;
    if (units == 0) return 0;
    if (units > (int64_t)0x7fffffff) return (int)cudaErrorInvalidValue;
    GradParams prm{};
    prm.chunks = c->dev.wy_chunks;
    prm.q = (const __nv_bfloat16 *)q;
    prm.k = (const __nv_bfloat16 *)k;
    prm.v = (const __nv_bfloat16 *)v;
    prm.beta = (const __nv_bfloat16 *)beta;
    prm.dout = (const __nv_bfloat16 *)dout;
    prm.g = g;
    prm.T = tmat;
    prm.S = st_S;
    prm.Dl = st_D;
    prm.dS = st_dS;
    prm.dD = st_dD;
    prm.dq = dq;
    prm.dk = dk;
    prm.dv = dv;
    prm.dbeta = dbeta;
    prm.dg = dg;
    prm.H = pl.H;
    prm.G = pl.G;
    prm.scale = pl.scale;
    auto kern = pl.G > 1 ? bwd_grad_kernel<true> : bwd_grad_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return (int)e;
    kern<<<(unsigned)units, NT, SMEM, (cudaStream_t)stream>>>(prm);
    return (int)cudaGetLastError();
}

}  // namespace cpdr
