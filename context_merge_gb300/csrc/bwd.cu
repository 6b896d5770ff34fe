// Backward of the segmented delta-rule forward on CUDA cores (fp32): the
// gradients of sum <do, o> + sum <dht, S_final> with respect to q, k, v,
// beta and the gates, organised as the article "flash-linear-attention
// 上下文并行CP ..." ([FLA-CP]) organises its backward (§2.2, §4: pre-process
// of the backward, the merge run in reverse with the transposed transfer
// matrices, then the state-gradient chains):
//   1. every segment's first fragment that continues a sequence runs the
//      reverse chain from its local end gradient (dht where the sequence
//      ends in it, else zero) and keeps the state gradient at its start,
//      dS_ext (the pre-process of the backward);
//   2. per sequence crossing cuts, the reverse merge
//      G = dS_ext[r1];  for j = r1-1 .. r0+1:  G <- M_j^T G + dS_ext[j],
//      giving the gradient at the end of every segment's continuing last
//      fragment (dS_end);
//   3. every fragment runs the reverse chain from dht (sequence ends in it),
//      dS_end (continues) or zero, and emits the input gradients.
// The chain is the reverse of the per-token update (the chain rule written
// out): with P = Diag(alpha) S_{t-1}, u = v - P^T k and G = dL/dS_t,
//   G += scale q do^T,  dq = scale S_t do,  g_u = beta G^T k,  dv = g_u,
//   dbeta = k^T G u,  dk = beta G u - P g_u,  dP = G - k g_u^T,
//   dg = alpha * sum_c dP S_{t-1} (per key dim; summed for a scalar gate),
//   dL/dS_{t-1} = Diag(alpha) dP.
// With grouped query heads (Hq = G H, [FLA-CP] §5.1) the first line runs
// for each of the state's G query heads: G += scale q_g do_g^T and
// dq_g = scale S_t do_g.
// The forward states are recomputed per token: from S_init (or zero) the
// chain first stores the state at every 64-token boundary, then walks the
// chunks backwards, recomputing each chunk's states into a per-CTA scratch.
// A chunk's token vectors are staged in shared memory at once, so the token
// steps read no global memory; only the reverse pass's sums over the value
// columns need a block barrier per token.
//
// One CTA = one (fragment, head, 32-value-column tile), persistent over the
// work list.  A thread holds D/8 rows of one column (column = thread / 8),
// so reductions over the key dim are 8-lane shuffles; reductions over the
// value columns (dq, dk, dg, dbeta) go through shared memory and then
// atomically into the fp32 outputs, which the caller zeroes first.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cpdr_internal.hpp"

namespace cpdr {
namespace {

constexpr int BT = 256;     // threads per CTA
constexpr int BVT = 32;     // value columns per CTA
constexpr int CKB = 64;     // tokens between checkpoints


struct BwdParams {
    const cpdr_fragment *frags;
    const int32_t *items;     // fragment indices of this pass
    int n_items;
    int mode;                 // 0: pre-process (dS_ext only), 1: main (input gradients)
    int H, B;
    int G;                    // query heads per state (q, do, dq have G H heads)
    int vfirst;               // S_init and dht stored [dv][dk]
    float scale;
    const void *q, *k, *v, *beta, *dout;
    const float *g;
    const float *dht;         // [N, H, D, D] or null
    const float *S_init;      // [R, B, H, D, D]
    const float *dS_end;      // [R, B, H, D, D] (main)
    float *dS_ext;            // [R, B, H, D, D] (pre-process)
    float *dq, *dk, *dv, *dbeta, *dg;
    float *scratch;           // per CTA: ckpt_floats + CKB * D * BVT floats
    int64_t ckpt_floats;      // max checkpoints per fragment * D * BVT
};

// Shared memory of one chunk's token vectors (raw input types; the gate as
// alpha = e^g in fp32), then the per-warp partial sums of the reverse pass.
// The query-head parts follow the struct, one block per query head of the
// state: q rows [G][CKB][D], do columns [G][CKB][BVT], and the partial sums
// [8 warps][2 + G][D] (dk, dalpha, then dq of each query head).
template <typename TIn, int D, bool PERDIM>
struct BwdSmem {
    static constexpr int NA = PERDIM ? D : 1;
    TIn kc[CKB][D], vc[CKB][BVT];
    float ac[CKB][NA], bc[CKB];
    float redb[8];
};
template <typename TIn, int D, bool PERDIM>
constexpr size_t bwd_smem_bytes(int G) {
    return (sizeof(BwdSmem<TIn, D, PERDIM>) + 15) / 16 * 16 + (size_t)G * CKB * D * sizeof(TIn) +
           (size_t)G * CKB * BVT * sizeof(TIn) + (size_t)8 * (2 + G) * D * sizeof(float);
}

__device__ __forceinline__ float tof(float x) { return x; }
__device__ __forceinline__ float tof(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename TIn, int D, bool PERDIM>
__global__ void __launch_bounds__(BT, 2) bwd_chain_kernel(const __grid_constant__ BwdParams p) {
    constexpr int NR = D / 8;                      // rows per thread
    extern __shared__ __align__(16) uint8_t bsm[];
    BwdSmem<TIn, D, PERDIM> &sm = *reinterpret_cast<BwdSmem<TIn, D, PERDIM> *>(bsm);
    const int GQ = p.G, Hq = p.H * GQ;
    TIn *qc = reinterpret_cast<TIn *>(bsm + (sizeof(BwdSmem<TIn, D, PERDIM>) + 15) / 16 * 16);   // [G][CKB][D]
    TIn *dc = qc + (size_t)GQ * CKB * D;                                                          // [G][CKB][BVT]
    float *red = reinterpret_cast<float *>(dc + (size_t)GQ * CKB * BVT);                          // [8][2 + G][D]
    auto redp = [&](int ww, int which) { return red + ((size_t)ww * (2 + GQ) + which) * D; };
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = tid >> 3, r8 = tid & 7;          // column in the tile, row group
    const int ntile = D / BVT;
    const TIn *q = (const TIn *)p.q, *k = (const TIn *)p.k, *v = (const TIn *)p.v, *beta = (const TIn *)p.beta,
              *dout = (const TIn *)p.dout;
    float *ck = p.scratch + (int64_t)blockIdx.x * (p.ckpt_floats + (int64_t)CKB * D * BVT);
    float *tok = ck + p.ckpt_floats;
    for (int item = blockIdx.x; item < p.n_items * p.H * ntile; item += gridDim.x) {
        const int tile = item % ntile, h = (item / ntile) % p.H;
        const cpdr_fragment f = p.frags[p.items[item / (ntile * p.H)]];
        const int col = tile * BVT + c;            // value dim of this thread
        const int64_t sidx = ((int64_t)f.seg * p.H + h) * D * D;
        // all token vectors of tokens [t0, t0 + nb) into shared memory, every
        // load independent (one latency per chunk); q and do for the reverse
        auto stage = [&](int t0, int nb, bool with_q) {
            __syncthreads();   // the previous chunk's readers are done
            for (int e = tid; e < nb * D; e += BT) {
                const int i = e / D, d = e % D;
                const int64_t th = (f.tok0 + t0 + i) * p.H + h;
                sm.kc[i][d] = k[th * D + d];
                if (PERDIM) sm.ac[i][d] = exp2f(p.g[th * D + d] * 1.4426950408889634f);
            }
            if (with_q) {
                for (int e = tid; e < GQ * nb * D; e += BT) {
                    const int gq = e / (nb * D), i = (e / D) % nb, d = e % D;
                    const int64_t tq = (f.tok0 + t0 + i) * Hq + (int64_t)h * GQ + gq;
                    qc[((size_t)gq * CKB + i) * D + d] = q[tq * D + d];
                }
                for (int e = tid; e < GQ * nb * BVT; e += BT) {
                    const int gq = e / (nb * BVT), i = (e / BVT) % nb, cc = e % BVT;
                    const int64_t tq = (f.tok0 + t0 + i) * Hq + (int64_t)h * GQ + gq;
                    dc[((size_t)gq * CKB + i) * BVT + cc] = dout[tq * D + tile * BVT + cc];
                }
            }
            for (int e = tid; e < nb * BVT; e += BT) {
                const int i = e / BVT, cc = e % BVT;
                const int64_t th = (f.tok0 + t0 + i) * p.H + h;
                sm.vc[i][cc] = v[th * D + tile * BVT + cc];
            }
            for (int i = tid; i < nb; i += BT) {
                const int64_t th = (f.tok0 + t0 + i) * p.H + h;
                sm.bc[i] = tof(beta[th]);
                if (!PERDIM) sm.ac[i][0] = exp2f(p.g[th] * 1.4426950408889634f);
            }
            __syncthreads();
        };
        auto alpha = [&](int i, int d) -> float { return PERDIM ? sm.ac[i][d] : sm.ac[i][0]; };
        // one forward token (chunk row i) on the register state s
        auto fwd_tok = [&](float (&s)[NR], int i) {
            float pk = 0.f;
#pragma unroll
            for (int j = 0; j < NR; j++) {
                const int d = r8 + 8 * j;
                s[j] *= alpha(i, d);
                pk = fmaf(s[j], tof(sm.kc[i][d]), pk);
            }
            pk += __shfl_xor_sync(0xffffffffu, pk, 1);
            pk += __shfl_xor_sync(0xffffffffu, pk, 2);
            pk += __shfl_xor_sync(0xffffffffu, pk, 4);
            const float bu = sm.bc[i] * (tof(sm.vc[i][c]) - pk);
#pragma unroll
            for (int j = 0; j < NR; j++) s[j] = fmaf(tof(sm.kc[i][r8 + 8 * j]), bu, s[j]);
        };
        // ---- forward: checkpoints at every 64-token boundary
        float s[NR];
#pragma unroll
        for (int j = 0; j < NR; j++)
            s[j] = (f.flags & CPDR_FRAG_CONT_PREV)
                       ? p.S_init[sidx + (p.vfirst ? (int64_t)col * D + r8 + 8 * j : (int64_t)(r8 + 8 * j) * D + col)]
                       : 0.f;
        const int nck = (f.len + CKB - 1) / CKB;
        for (int m = 0; m < nck; m++) {
            const int t0 = m * CKB, nb = min(CKB, f.len - t0);
#pragma unroll
            for (int j = 0; j < NR; j++) ck[((int64_t)m * BT + tid) * NR + j] = s[j];
            stage(t0, nb, false);
            for (int i = 0; i < nb; i++) fwd_tok(s, i);
        }
        // ---- the end gradient
        float G[NR];
        {
            const float *src = nullptr;
            int64_t base = 0;
            bool tr = false;   // dht in the [dv][dk] layout
            if (f.flags & CPDR_FRAG_ENDS_SEQ) {
                if (p.dht) { src = p.dht; base = ((int64_t)f.seq * p.H + h) * D * D; tr = p.vfirst != 0; }
            } else if ((f.flags & CPDR_FRAG_CONT_NEXT) && p.mode == 1) {
                src = p.dS_end;
                base = sidx;
            }
#pragma unroll
            for (int j = 0; j < NR; j++)
                G[j] = src ? src[base + (tr ? (int64_t)col * D + r8 + 8 * j : (int64_t)(r8 + 8 * j) * D + col)] : 0.f;
        }
        // ---- reverse over the chunks
        for (int m = nck - 1; m >= 0; m--) {
            const int t0 = m * CKB, nb = min(CKB, f.len - t0);
            stage(t0, nb, true);
#pragma unroll
            for (int j = 0; j < NR; j++) s[j] = ck[((int64_t)m * BT + tid) * NR + j];
            for (int i = 0; i < nb; i++) {   // the chunk's states, before each token
#pragma unroll
                for (int j = 0; j < NR; j++) tok[((int64_t)i * BT + tid) * NR + j] = s[j];
                fwd_tok(s, i);
            }
            // s = state after the chunk's last token; the state before token i
            // is loaded one token ahead (spn), hiding the scratch latency
            float spn[NR];
#pragma unroll
            for (int j = 0; j < NR; j++) spn[j] = tok[((int64_t)(nb - 1) * BT + tid) * NR + j];
            for (int i = nb - 1; i >= 0; i--) {
                const int64_t th = (f.tok0 + t0 + i) * p.H + h;
                float sp[NR];
#pragma unroll
                for (int j = 0; j < NR; j++) sp[j] = spn[j];
                if (i > 0) {
#pragma unroll
                    for (int j = 0; j < NR; j++) spn[j] = tok[((int64_t)(i - 1) * BT + tid) * NR + j];
                }
                const float bt = sm.bc[i];
                if (p.mode == 1) __syncthreads();   // the previous token's sums were read
                // per query head: dq partial (S_t do), summed over the warp's
                // 4 columns into this warp's slot, and G += q do^T
                for (int gq = 0; gq < GQ; gq++) {
                    const float ddc = p.scale * tof(dc[((size_t)gq * CKB + i) * BVT + c]);
                    const TIn *qrow = qc + ((size_t)gq * CKB + i) * D;
                    float pdq[NR];
#pragma unroll
                    for (int j = 0; j < NR; j++) {
                        pdq[j] = s[j] * ddc;
                        G[j] = fmaf(tof(qrow[r8 + 8 * j]), ddc, G[j]);
                    }
                    if (p.mode == 1) {
#pragma unroll
                        for (int j = 0; j < NR; j++) {
#pragma unroll
                            for (int o = 8; o < 32; o <<= 1) pdq[j] += __shfl_xor_sync(0xffffffffu, pdq[j], o);
                        }
                        if (lane < 8) {
#pragma unroll
                            for (int j = 0; j < NR; j++) redp(w, 2 + gq)[lane + 8 * j] = pdq[j];
                        }
                    }
                }
                // P = Diag(alpha) S_{t-1}: P^T k and G^T k
                float pk = 0.f, gk = 0.f;
#pragma unroll
                for (int j = 0; j < NR; j++) {
                    const int d = r8 + 8 * j;
                    const float kd = tof(sm.kc[i][d]);
                    pk = fmaf(alpha(i, d) * sp[j], kd, pk);
                    gk = fmaf(G[j], kd, gk);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    pk += __shfl_xor_sync(0xffffffffu, pk, o);
                    gk += __shfl_xor_sync(0xffffffffu, gk, o);
                }
                const float u = tof(sm.vc[i][c]) - pk, gu = bt * gk;
                if (p.mode == 1 && r8 == 0) p.dv[th * D + col] = gu;
                // dk partial, dalpha partial, dbeta partial; then G <- Diag(alpha) dP
                float pdk[NR], pda[NR], pb = 0.f;
#pragma unroll
                for (int j = 0; j < NR; j++) {
                    const int d = r8 + 8 * j;
                    const float kd = tof(sm.kc[i][d]), al = alpha(i, d);
                    const float Gu = G[j] * u;
                    pb = fmaf(kd, Gu, pb);
                    pdk[j] = bt * Gu - al * sp[j] * gu;
                    const float dP = G[j] - kd * gu;
                    pda[j] = dP * sp[j];             // dP * S_{t-1}
                    G[j] = al * dP;
                }
                if (p.mode == 1) {
                    // sum over the warp's 4 columns, then across the 8 warps
#pragma unroll
                    for (int j = 0; j < NR; j++) {
#pragma unroll
                        for (int o = 8; o < 32; o <<= 1) {
                            pdk[j] += __shfl_xor_sync(0xffffffffu, pdk[j], o);
                            pda[j] += __shfl_xor_sync(0xffffffffu, pda[j], o);
                        }
                    }
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
                    if (lane < 8) {
#pragma unroll
                        for (int j = 0; j < NR; j++) {
                            redp(w, 0)[lane + 8 * j] = pdk[j];
                            redp(w, 1)[lane + 8 * j] = pda[j];
                        }
                    }
                    if (lane == 0) sm.redb[w] = pb;
                    __syncthreads();
                    float dgs = 0.f;   // scalar gate: this thread's share of sum_d alpha dalpha
                    const int64_t tqd = ((f.tok0 + t0 + i) * Hq + (int64_t)h * GQ) * D;   // dq of query head 0
                    for (int e = tid; e < (2 + GQ) * D; e += BT) {
                        const int which = e / D, d = e % D;
                        float acc = 0.f;
#pragma unroll
                        for (int ww = 0; ww < 8; ww++) acc += redp(ww, which)[d];
                        if (which == 0) atomicAdd(p.dk + th * D + d, acc);
                        else if (which == 1) {
                            if (PERDIM) atomicAdd(p.dg + th * D + d, alpha(i, d) * acc);
                            else dgs += alpha(i, d) * acc;
                        } else {
                            atomicAdd(p.dq + tqd + (int64_t)(which - 2) * D + d, acc);
                        }
                    }
                    if (tid == 0) {
                        float acc = 0.f;
#pragma unroll
                        for (int ww = 0; ww < 8; ww++) acc += sm.redb[ww];
                        atomicAdd(p.dbeta + th, acc);
                    }
                    if (!PERDIM) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) dgs += __shfl_xor_sync(0xffffffffu, dgs, o);
                        if (lane == 0 && dgs != 0.f) atomicAdd(p.dg + th, dgs);
                    }
                }
                // the state before this token is the next one's S_t
#pragma unroll
                for (int j = 0; j < NR; j++) s[j] = sp[j];
            }
        }
        // ---- the pre-process keeps the gradient at the fragment start
        if (p.mode == 0) {
#pragma unroll
            for (int j = 0; j < NR; j++) p.dS_ext[sidx + (int64_t)(r8 + 8 * j) * D + col] = G[j];
        }
    }
}

// Reverse merge: grid (chains, H, D / BVT); thread = rows r8 + 8 i of one column.
template <int D>
__global__ void __launch_bounds__(BT) bwd_merge_kernel(const MergeChain *__restrict__ chains,
                                                       const float *__restrict__ dS_ext, const float *__restrict__ M,
                                                       float *__restrict__ dS_end, int H, int B) {
    constexpr int NR = D / 8;
    __shared__ float Gs[D][BVT + 1];
    const MergeChain ch = chains[blockIdx.x];
    const int h = blockIdx.y, tile = blockIdx.z;
    const int c = threadIdx.x >> 3, r8 = threadIdx.x & 7, col = tile * BVT + c;
    auto idx_of = [&](int r) { return ((int64_t)(r * B + ch.b) * H + h) * D * D; };
    float G[NR];
#pragma unroll
    for (int i = 0; i < NR; i++) {
        G[i] = dS_ext[idx_of(ch.r1) + (int64_t)(r8 + 8 * i) * D + col];
        dS_end[idx_of(ch.r1 - 1) + (int64_t)(r8 + 8 * i) * D + col] = G[i];
    }
    for (int j = ch.r1 - 1; j > ch.r0; j--) {
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NR; i++) Gs[r8 + 8 * i][c] = G[i];
        __syncthreads();
        const float *Mj = M + idx_of(j);
#pragma unroll
        for (int i = 0; i < NR; i++) {
            const int d = r8 + 8 * i;
            float acc = dS_ext[idx_of(j) + (int64_t)d * D + col];
            for (int l = 0; l < D; l++) acc = fmaf(__ldg(Mj + (int64_t)l * D + d), Gs[l][c], acc);   // (M^T G)[d]
            G[i] = acc;
            dS_end[idx_of(j - 1) + (int64_t)d * D + col] = acc;
        }
    }
}

template <typename TIn, int D, bool PERDIM>
int launch_chain_t(const BwdParams &prm, int grid, cudaStream_t st) {
    const size_t sm = bwd_smem_bytes<TIn, D, PERDIM>(prm.G);
    cudaError_t e = cudaFuncSetAttribute(bwd_chain_kernel<TIn, D, PERDIM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    bwd_chain_kernel<TIn, D, PERDIM><<<grid, BT, sm, st>>>(prm);
    return (int)cudaGetLastError();
}

template <int D>
int dispatch_chain(const cpdr_ctx *c, const BwdParams &prm, int grid, cudaStream_t st) {
    const bool perdim = c->plan.gate_kind == CPDR_GATE_PER_DIM;
    if (c->plan.in_dtype == CPDR_DTYPE_F32)
        return perdim ? launch_chain_t<float, D, true>(prm, grid, st) : launch_chain_t<float, D, false>(prm, grid, st);
    return perdim ? launch_chain_t<__nv_bfloat16, D, true>(prm, grid, st)
                  : launch_chain_t<__nv_bfloat16, D, false>(prm, grid, st);
}

}  // namespace

int bwd_grid(const cpdr_ctx *c) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int64_t work = (int64_t)c->plan.frags.size() * c->plan.H * (c->plan.dk / BVT);
    return (int)std::max<int64_t>(1, std::min<int64_t>(work, (int64_t)sms * 4));
}

size_t bwd_scratch_floats_per_cta(const cpdr_ctx *c) {
    const auto &p = c->plan;
    int32_t maxlen = 0;
    for (const auto &f : p.frags) maxlen = std::max(maxlen, f.len);
    const int64_t nck = (maxlen + CKB - 1) / CKB;
    return (size_t)(nck + CKB) * p.dk * BVT;
}

// Whether the CUDA-core chain's shared memory holds the G query heads' rows
// of one chunk.
bool bwd_simt_fits(const cpdr_ctx *c) {
    const auto &p = c->plan;
    const int G = p.Hq / p.H;
    const bool f32 = p.in_dtype == CPDR_DTYPE_F32, perdim = p.gate_kind == CPDR_GATE_PER_DIM;
    size_t need;
    if (p.dk == 64)
        need = f32 ? (perdim ? bwd_smem_bytes<float, 64, true>(G) : bwd_smem_bytes<float, 64, false>(G))
                   : (perdim ? bwd_smem_bytes<__nv_bfloat16, 64, true>(G) : bwd_smem_bytes<__nv_bfloat16, 64, false>(G));
    else
        need = f32 ? (perdim ? bwd_smem_bytes<float, 128, true>(G) : bwd_smem_bytes<float, 128, false>(G))
                   : (perdim ? bwd_smem_bytes<__nv_bfloat16, 128, true>(G)
                             : bwd_smem_bytes<__nv_bfloat16, 128, false>(G));
    return need <= 232448;
}

// bf16, d = 128: both gates, grouped query heads and both state layouts
bool bwd_uses_tc(const cpdr_ctx *c) { return c->use_tc; }

namespace {
size_t r256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

// Scratch of the tensor-core backward: the WY tiles, then per (chunk, head)
// the chunk's starting state S and Delta (recomputed) and the state-gradient
// chain's dS' and dDelta (fp32).
size_t bwd_tc_scratch_bytes(const cpdr_ctx *c) {
    const auto &p = c->plan;
    const size_t units = p.wy_chunks.size() * (size_t)p.H;
    const size_t st = units * (size_t)p.dk * p.dv * sizeof(float), dl = units * 64 * (size_t)p.dv * sizeof(float);
    return r256(wy_bytes(c)) + r256(units * 64 * 64 * sizeof(float)) + 2 * r256(st) + 2 * r256(dl);
}

// The backward on the tensor cores ([FLA-CP] §2.2, §4): the WY tiles; the
// forward recomputed with every chunk's starting state and Delta stored;
// the state-gradient chains of the segments' first continuing fragments
// (dS_ext); the reverse merge (dS_end); the state-gradient chains of every
// fragment, storing dS' and dDelta per chunk; the input gradients of every
// (chunk, head) in parallel.
int launch_bwd_tc(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta, const float *g,
                  const void *dout, const float *dht, const float *S_init, const float *M, float *dS_ext,
                  float *dS_end, void *scratch, float *dq, float *dk, float *dv, float *dbeta, float *dg,
                  void *stream) {
    const auto &p = c->plan;
    const size_t units = p.wy_chunks.size() * (size_t)p.H;
    const size_t stb = units * (size_t)p.dk * p.dv * sizeof(float), dlb = units * 64 * (size_t)p.dv * sizeof(float);
    char *w = (char *)scratch;
    void *wy = w;
    w += r256(wy_bytes(c));
    float *tmat = (float *)w;
    w += r256(units * 64 * 64 * sizeof(float));
    float *st_S = (float *)w;
    w += r256(stb);
    float *st_dS = (float *)w;
    w += r256(stb);
    float *st_D = (float *)w;
    w += r256(dlb);
    float *st_dD = (float *)w;
    const bool kda = p.gate_kind == CPDR_GATE_PER_DIM;
    int rc = kda ? launch_tc_kda_prep_t(c, k, q, beta, g, wy, tmat, stream)
                 : launch_tc_wy_t(c, k, beta, g, wy, tmat, stream);
    if (rc) return rc;
    rc = launch_tc_rec(c, k, v, g, wy, S_init, st_S, st_D, stream);
    if (rc) return rc;
    // the state-gradient chains once per query head of a state (the first
    // pass writes, the others add: the chain is linear in its q, dO terms)
    if (!p.bwd_pre_items.empty()) {
        for (int gq = 0; gq < p.G && !rc; gq++)
            rc = launch_tc_bwd_chain(c, c->dev.bwd_pre_items, (int)p.bwd_pre_items.size(), 1, gq, q, k, dout, g, wy,
                                     dht, nullptr, dS_ext, nullptr, nullptr, stream);
        if (rc) return rc;
    }
    rc = launch_tc_merge_rev(c, dS_ext, M, dS_end, stream);
    if (rc) return rc;
    for (int gq = 0; gq < p.G && !rc; gq++)
        rc = launch_tc_bwd_chain(c, c->dev.fwd_order, (int)p.frags.size(), 0, gq, q, k, dout, g, wy, dht, dS_end,
                                 nullptr, st_dS, st_dD, stream);
    if (rc) return rc;
    if (kda)
        return launch_bwd_grad_kda(c, q, k, v, beta, g, dout, tmat, st_S, st_D, st_dS, st_dD, dq, dk, dv, dbeta, dg,
                                   stream);
    return launch_bwd_grad(c, q, k, v, beta, g, dout, tmat, st_S, st_D, st_dS, st_dD, dq, dk, dv, dbeta, dg,
                           stream);
}

int launch_bwd(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta, const float *g,
               const void *dout, const float *dht, const float *S_init, const float *M, float *dS_ext,
               float *dS_end, float *scratch, float *dq, float *dk, float *dv, float *dbeta, float *dg,
               void *stream) {
    if (bwd_uses_tc(c))
        return launch_bwd_tc(c, q, k, v, beta, g, dout, dht, S_init, M, dS_ext, dS_end, scratch, dq, dk, dv, dbeta,
                             dg, stream);
    cudaStream_t st = (cudaStream_t)stream;
    const auto &p = c->plan;
    BwdParams prm{};
    prm.frags = c->dev.frags;
    prm.H = p.H;
    prm.B = p.B;
    prm.G = p.Hq / p.H;
    prm.vfirst = p.vfirst ? 1 : 0;
    prm.scale = p.scale;
    prm.q = q; prm.k = k; prm.v = v; prm.beta = beta; prm.dout = dout; prm.g = g;
    prm.dht = dht; prm.S_init = S_init; prm.dS_end = dS_end; prm.dS_ext = dS_ext;
    prm.dq = dq; prm.dk = dk; prm.dv = dv; prm.dbeta = dbeta; prm.dg = dg;
    prm.scratch = scratch;
    prm.ckpt_floats = (int64_t)bwd_scratch_floats_per_cta(c) - (int64_t)CKB * p.dk * BVT;
    const int grid = bwd_grid(c);
    int rc = 0;
    // 1. the pre-process: segments' first fragments that continue a sequence
    if (!p.bwd_pre_items.empty()) {
        prm.items = c->dev.bwd_pre_items;
        prm.n_items = (int)p.bwd_pre_items.size();
        prm.mode = 0;
        rc = p.dk == 64 ? dispatch_chain<64>(c, prm, grid, st) : dispatch_chain<128>(c, prm, grid, st);
        if (rc) return rc;
    }
    // 2. the reverse merge
    if (!p.chains.empty()) {
        dim3 mg((unsigned)p.chains.size(), (unsigned)p.H, (unsigned)(p.dk / BVT));
        if (p.dk == 64)
            bwd_merge_kernel<64><<<mg, BT, 0, st>>>(c->dev.chains, dS_ext, M, dS_end, p.H, p.B);
        else
            bwd_merge_kernel<128><<<mg, BT, 0, st>>>(c->dev.chains, dS_ext, M, dS_end, p.H, p.B);
        rc = (int)cudaGetLastError();
        if (rc) return rc;
    }
    // 3. every fragment, with its end gradient
    prm.items = c->dev.fwd_order;
    prm.n_items = (int)p.frags.size();
    prm.mode = 1;
    return p.dk == 64 ? dispatch_chain<64>(c, prm, grid, st) : dispatch_chain<128>(c, prm, grid, st);
}

}  // namespace cpdr
