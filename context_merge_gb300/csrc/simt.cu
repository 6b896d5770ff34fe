// fp32 CUDA-core kernels for the segmented delta-rule forward: the path for
// fp32 inputs and for d = 64, and a cross-check of the tensor-core path.
//
// Each kernel follows the chunk form of the article "flash-linear-attention
// 上下文并行CP ..." ([FLA-CP]), §2.2, with 64-token chunks, computed in fp32:
//   G   = in-chunk cumulative log2 gates (chunk_local_cumsum, scale 1/ln 2, §4)
//   A   = strictly lower, A_ij = beta_i sum_d k_id k_jd 2^(G_id - G_jd)
//   (I + A) [W | U] = [diag(beta)(gamma ⊙ K) | diag(beta) V]     (forward substitution)
//   Delta = U - W S                       ("v_new")
//   O     = scale [(gamma ⊙ Q) S + (Q K^T ⊙ Lambda) Delta]
//   S    <- Diag(gamma^C) S + (Gamma ⊙ K)^T Delta
// The pre-process runs the same chain on X = [S | M] with X_0 = [0 | I] and
// the M columns' U equal to zero, which is M <- M_[t] M with
// M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W (§2.1-§2.2).
//
// One CTA owns one (fragment, head, 32-column tile) chain; padded rows of a
// partial chunk carry k = v = q = beta = g = 0, which is the identity map.
// For the per-dim gate (KDA) the exponentials are factored around the
// chunk's middle row r: 2^(G_i - G_j) = 2^(G_i - G_r) 2^(G_r - G_j), each
// factor bounded by the decay over half a chunk.  A chunk whose decay
// exceeds 2^100 either way of row r (where a factor could overflow) takes
// exact per-term exponentials for A and Q K^T instead, and the unfactored
// forms k 2^G, q 2^G, k 2^(G_C - G) for the rest.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"

namespace cpdr {
namespace {

constexpr int C = kChunk;     // 64
constexpr int BV = 32;        // state columns per CTA
constexpr int NT = 256;       // threads per CTA
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ldf(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void stf(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// Offset of state element (key dim d, value dim c) inside one D x D state:
// [dk][dv] by default, [dv][dk] in the state_v_first layout.
template <int D>
__device__ __forceinline__ int64_t st_off(int d, int c, bool vfirst) {
    return vfirst ? (int64_t)c * D + d : (int64_t)d * D + c;
}

// Shared-memory layout of one chunk (row strides padded by one float).
template <int D>
struct Smem {
    static constexpr int LD = D + 1;     // row stride of [C][D] tiles
    static constexpr int LA = C + 1;     // row stride of [C][C] tiles
    static constexpr int LB = BV + 1;    // row stride of [*][BV] tiles
    float Ki[C * LD];      // GDN: k;  KDA: k * 2^(G - G_ref)
    float Kj[C * LD];      // KDA only: k * 2^(G_ref - G)
    float Qi[C * LD];      // GDN: q;  KDA: q * 2^(G - G_ref)
    float A[C * LA];       // strictly lower A (then kept for nothing else)
    float QK[C * LA];      // lower (incl. diagonal) Q K^T ⊙ Lambda
    float WU[C * (D + BV + 1)];   // [W | U] after the solve
    float S[D * LB];       // state tile (D x BV)
    float Dl[C * LB];      // Delta
    float g1[C];           // GDN: cumulative log2 gate per row
    float gref[D], gC[D];  // KDA: G at the reference row (0 when exact) and at the last row
    // KDA: the per-dim cumulative gates [C][LD] live in WU until the solve
    __device__ float *Gk() { return WU; }
    float beta[C];
    int exact;             // KDA: this chunk takes exact per-term exponentials
};

constexpr float kFactorBound = 100.f;   // largest |G_i - G_r| (log2) of the factored form

template <int D>
constexpr size_t smem_bytes() { return sizeof(Smem<D>); }

// Load one chunk (rows >= n zero-filled) and build the gate factors.
template <typename TIn, int D, bool PERDIM>
__device__ void load_chunk(Smem<D> &s, const TIn *q, const TIn *k, const TIn *beta, const float *g,
                           int64_t tok0, int n, int H, int h, int Hq, int hq) {
    constexpr int LD = Smem<D>::LD;
    const int tid = threadIdx.x;
    for (int idx = tid; idx < C * D; idx += NT) {
        const int i = idx / D, d = idx % D;
        float kv = 0.f, qv = 0.f, gv = 0.f;
        if (i < n) {
            const int64_t off = ((tok0 + i) * H + h) * (int64_t)D + d;
            kv = ldf(k, off);
            if (q) qv = ldf(q, ((tok0 + i) * Hq + hq) * (int64_t)D + d);
            if (PERDIM) gv = g[off] * kLog2e;
        }
        s.Ki[i * LD + d] = kv;
        s.Qi[i * LD + d] = qv;
        if (PERDIM) s.Gk()[i * LD + d] = gv;
    }
    for (int i = tid; i < C; i += NT) {
        float b = 0.f, gv = 0.f;
        if (i < n) {
            b = ldf(beta, (tok0 + i) * H + h);
            if (!PERDIM) gv = g[(tok0 + i) * H + h] * kLog2e;
        }
        s.beta[i] = b;
        if (!PERDIM) s.g1[i] = gv;
    }
    __syncthreads();
    // in-chunk cumulative sums (one thread per gate column)
    int far = 0;
    if (PERDIM) {
        for (int d = tid; d < D; d += NT) {
            float acc = 0.f;
            for (int i = 0; i < C; i++) { acc += s.Gk()[i * LD + d]; s.Gk()[i * LD + d] = acc; }
            const float gr = s.Gk()[(C / 2 - 1) * LD + d];
            for (int i = 0; i < C; i++) far |= fabsf(s.Gk()[i * LD + d] - gr) > kFactorBound;
            s.gref[d] = gr;
            s.gC[d] = acc;
        }
    } else if (tid < 32) {
        // warp scan over 64 scalars, two per lane
        float a0 = s.g1[2 * tid], a1 = s.g1[2 * tid + 1];
        float x = a0 + a1;
        for (int o = 1; o < 32; o <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, x, o);
            if (tid >= o) x += y;
        }
        const float excl = x - (a0 + a1);
        s.g1[2 * tid] = excl + a0;
        s.g1[2 * tid + 1] = x;
    }
    const int exact = __syncthreads_or(far);
    if (tid == 0) s.exact = exact;
    if (PERDIM && !exact) {
        for (int idx = tid; idx < C * D; idx += NT) {
            const int i = idx / D, d = idx % D;
            const float gi = s.Gk()[i * LD + d], gr = s.gref[d];
            const float kv = s.Ki[i * LD + d];
            s.Kj[i * LD + d] = kv * exp2f(gr - gi);
            s.Ki[i * LD + d] = kv * exp2f(gi - gr);
            s.Qi[i * LD + d] = s.Qi[i * LD + d] * exp2f(gi - gr);
        }
    }
    __syncthreads();
}

// Per-dim gate, exact branch: A_ij = beta_i sum_d k_id k_jd 2^(G_id - G_jd)
// (j < i) and Q K^T ⊙ Lambda with one exponential per term (Ki, Qi hold k
// and q; the cumulative gates are still in WU); then the tiles take the
// unfactored forms Ki = k 2^G, Qi = q 2^G, Kj = k 2^(G_C - G) and gref = 0.
template <int D, bool WITH_Q>
__device__ void build_A_QK_exact(Smem<D> &s) {
    constexpr int LD = Smem<D>::LD, LA = Smem<D>::LA;
    const int tid = threadIdx.x;
    const int j = tid % C, ib = tid / C;   // 4 blocks of 16 rows
    const float *Gk = s.Gk();
    float acc[16], accq[16];
#pragma unroll
    for (int r = 0; r < 16; r++) { acc[r] = 0.f; accq[r] = 0.f; }
    for (int d = 0; d < D; d++) {
        const float kj = s.Ki[j * LD + d], gj = Gk[j * LD + d];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            const int i = ib * 16 + r;
            if (j > i) continue;
            const float lam = exp2f(Gk[i * LD + d] - gj) * kj;
            acc[r] = fmaf(s.Ki[i * LD + d], lam, acc[r]);
            if (WITH_Q) accq[r] = fmaf(s.Qi[i * LD + d], lam, accq[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < 16; r++) {
        const int i = ib * 16 + r;
        s.A[i * LA + j] = (j < i) ? s.beta[i] * acc[r] : 0.f;
        if (WITH_Q) s.QK[i * LA + j] = (j <= i) ? accq[r] : 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < C * D; idx += NT) {
        const int i = idx / D, d = idx % D;
        const float gi = Gk[i * LD + d], kv = s.Ki[i * LD + d];
        s.Kj[i * LD + d] = kv * exp2f(s.gC[d] - gi);
        s.Ki[i * LD + d] = kv * exp2f(gi);
        s.Qi[i * LD + d] = s.Qi[i * LD + d] * exp2f(gi);
    }
    for (int d = tid; d < D; d += NT) s.gref[d] = 0.f;
}

// A (strictly lower, scaled by beta_i) and QK ⊙ Lambda (lower incl. diagonal).
template <int D, bool PERDIM, bool WITH_Q>
__device__ void build_A_QK(Smem<D> &s) {
    constexpr int LD = Smem<D>::LD, LA = Smem<D>::LA;
    const int tid = threadIdx.x;
    const int j = tid % C, ib = tid / C;   // 4 blocks of 16 rows
    const float *Kjs = PERDIM ? s.Kj : s.Ki;
    float acc[16], accq[16];
#pragma unroll
    for (int r = 0; r < 16; r++) { acc[r] = 0.f; accq[r] = 0.f; }
    if (PERDIM && s.exact) {
        build_A_QK_exact<D, WITH_Q>(s);
        return;
    }
    for (int d = 0; d < D; d++) {
        const float kj = Kjs[j * LD + d];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            const int i = ib * 16 + r;
            acc[r] = fmaf(s.Ki[i * LD + d], kj, acc[r]);
            if (WITH_Q) accq[r] = fmaf(s.Qi[i * LD + d], kj, accq[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < 16; r++) {
        const int i = ib * 16 + r;
        float lam = 1.f;
        if (!PERDIM) lam = exp2f(s.g1[i] - s.g1[j]);
        s.A[i * LA + j] = (j < i) ? s.beta[i] * lam * acc[r] : 0.f;
        if (WITH_Q) s.QK[i * LA + j] = (j <= i) ? lam * accq[r] : 0.f;
    }
}

// Forward substitution of (I + A) [W | U] = rhs, one thread per column.
// Columns 0..D-1: rhs = beta_i gamma_i ⊙ k_i; columns D..D+BV-1: beta_i v_i
// (or zero for the M columns of the pre-process).
template <typename TIn, int D, bool PERDIM>
__device__ void solve_WU(Smem<D> &s, const TIn *v, int64_t tok0, int n, int H, int h, int vcol0,
                         bool v_zero) {
    constexpr int LD = Smem<D>::LD, LA = Smem<D>::LA, LW = D + BV + 1;
    const int c = threadIdx.x;
    if (c < D + BV) {
        // right-hand side
        for (int i = 0; i < C; i++) {
            float r;
            if (c < D) {
                const float gfac = PERDIM ? exp2f(s.gref[c]) : exp2f(s.g1[i]);
                r = s.beta[i] * s.Ki[i * LD + c] * gfac;
            } else {
                const int e = vcol0 + (c - D);
                r = (!v_zero && i < n) ? s.beta[i] * ldf(v, ((tok0 + i) * H + h) * (int64_t)(D) + e) : 0.f;
            }
            s.WU[i * LW + c] = r;
        }
        for (int i = 1; i < C; i++) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            int j = 0;
            for (; j + 4 <= i; j += 4) {
                a0 = fmaf(s.A[i * LA + j], s.WU[j * LW + c], a0);
                a1 = fmaf(s.A[i * LA + j + 1], s.WU[(j + 1) * LW + c], a1);
                a2 = fmaf(s.A[i * LA + j + 2], s.WU[(j + 2) * LW + c], a2);
                a3 = fmaf(s.A[i * LA + j + 3], s.WU[(j + 3) * LW + c], a3);
            }
            for (; j < i; j++) a0 = fmaf(s.A[i * LA + j], s.WU[j * LW + c], a0);
            s.WU[i * LW + c] -= (a0 + a1) + (a2 + a3);
        }
    }
}

// Delta = U - W S  (C x BV)
template <int D>
__device__ void delta_step(Smem<D> &s) {
    constexpr int LB = Smem<D>::LB, LW = D + BV + 1;
    const int c = threadIdx.x % BV, ib = threadIdx.x / BV;   // 8 blocks of 8 rows
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; r++) acc[r] = s.WU[(ib * 8 + r) * LW + D + c];
    for (int d = 0; d < D; d++) {
        const float sv = s.S[d * LB + c];
#pragma unroll
        for (int r = 0; r < 8; r++) acc[r] = fmaf(-s.WU[(ib * 8 + r) * LW + d], sv, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 8; r++) s.Dl[(ib * 8 + r) * LB + c] = acc[r];
}

// O = scale [(gamma ⊙ Q) S + (QK ⊙ Lambda) Delta], stored for valid rows
template <typename TIn, int D, bool PERDIM>
__device__ void output_step(Smem<D> &s, TIn *o, int64_t tok0, int n, int Hq, int hq, int vcol0,
                            float scale) {
    constexpr int LD = Smem<D>::LD, LA = Smem<D>::LA, LB = Smem<D>::LB;
    const int c = threadIdx.x % BV, ib = threadIdx.x / BV;
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; r++) acc[r] = 0.f;
    for (int d = 0; d < D; d++) {
        const float sv = s.S[d * LB + c] * (PERDIM ? exp2f(s.gref[d]) : 1.f);
#pragma unroll
        for (int r = 0; r < 8; r++) acc[r] = fmaf(s.Qi[(ib * 8 + r) * LD + d], sv, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 8; r++) {
        const int i = ib * 8 + r;
        float x = PERDIM ? acc[r] : acc[r] * exp2f(s.g1[i]);
        for (int j = 0; j <= i; j++) x = fmaf(s.QK[i * LA + j], s.Dl[j * LB + c], x);
        if (i < n) stf(o, ((tok0 + i) * Hq + hq) * (int64_t)D + vcol0 + c, scale * x);
    }
}

// S <- Diag(gamma^C) S + (Gamma ⊙ K)^T Delta
template <int D, bool PERDIM>
__device__ void state_step(Smem<D> &s, int n) {
    constexpr int LD = Smem<D>::LD, LB = Smem<D>::LB;
    const int c = threadIdx.x % BV, db = threadIdx.x / BV;   // 8 blocks of D/8 rows
    constexpr int RPT = D / 8;
    const float gC = PERDIM ? 0.f : s.g1[C - 1];
    float acc[RPT], cf[RPT];   // KDA: cf = 2^(G_C,d - G_ref,d), independent of the token
#pragma unroll
    for (int r = 0; r < RPT; r++) {
        const int d = db * RPT + r;
        acc[r] = s.S[d * LB + c] * exp2f(PERDIM ? s.gC[d] : gC);
        cf[r] = PERDIM ? (s.exact ? 1.f : exp2f(s.gC[d] - s.gref[d])) : 0.f;
    }
    for (int j = 0; j < C; j++) {
        const float dl = s.Dl[j * LB + c];
        const float gam = PERDIM ? 0.f : exp2f(gC - s.g1[j]);
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const int d = db * RPT + r;
            // KDA: Gamma_jd k_jd = Kj_jd * 2^(G_C,d - G_ref,d) (exact: Kj_jd)
            const float kg = PERDIM ? s.Kj[j * LD + d] * cf[r] : s.Ki[j * LD + d] * gam;
            acc[r] = fmaf(kg, dl, acc[r]);
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPT; r++) s.S[(db * RPT + r) * LB + c] = acc[r];
    (void)n;
}

// Forward: grid (fragments in fwd_order, Hq, dv / BV).  Query head hq runs
// the chain of state head h = hq / G (grouped query heads recompute it); the
// group's first query head writes the final state.
template <typename TIn, int D, bool PERDIM>
__global__ void __launch_bounds__(NT, 1)
simt_fwd_kernel(const cpdr_fragment *__restrict__ frags, const int32_t *__restrict__ order,
                const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                const TIn *__restrict__ beta, const float *__restrict__ g,
                const float *__restrict__ S_init, TIn *__restrict__ o, float *__restrict__ final_state,
                int H, int G, bool vfirst, float scale) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(smem_raw);
    constexpr int LB = Smem<D>::LB;
    const cpdr_fragment f = frags[order[blockIdx.x]];
    const int hq = blockIdx.y, h = hq / G, vcol0 = blockIdx.z * BV;
    // initial state (vfirst: consecutive threads walk the key dim, contiguous there)
    for (int idx = threadIdx.x; idx < D * BV; idx += NT) {
        const int d = vfirst ? idx % D : idx / BV, c = vfirst ? idx / D : idx % BV;
        float x = 0.f;
        if (f.flags & CPDR_FRAG_CONT_PREV)
            x = S_init[((int64_t)f.seg * H + h) * D * D + st_off<D>(d, vcol0 + c, vfirst)];
        s.S[d * LB + c] = x;
    }
    for (int c0 = 0; c0 < f.len; c0 += C) {
        const int n = min(C, f.len - c0);
        const int64_t t0 = f.tok0 + c0;
        __syncthreads();
        load_chunk<TIn, D, PERDIM>(s, q, k, beta, g, t0, n, H, h, H * G, hq);
        build_A_QK<D, PERDIM, true>(s);
        __syncthreads();
        solve_WU<TIn, D, PERDIM>(s, v, t0, n, H, h, vcol0, false);
        __syncthreads();
        delta_step<D>(s);
        __syncthreads();
        output_step<TIn, D, PERDIM>(s, o, t0, n, H * G, hq, vcol0, scale);
        state_step<D, PERDIM>(s, n);
    }
    __syncthreads();
    if ((f.flags & CPDR_FRAG_ENDS_SEQ) && final_state && hq % G == 0) {
        for (int idx = threadIdx.x; idx < D * BV; idx += NT) {
            const int d = vfirst ? idx % D : idx / BV, c = vfirst ? idx / D : idx % BV;
            final_state[((int64_t)f.seq * H + h) * D * D + st_off<D>(d, vcol0 + c, vfirst)] = s.S[d * LB + c];
        }
    }
}

// Pre-process: grid (pre items, H, 2 D / BV); column tiles < D/BV are S
// columns (U from v), the rest are M columns (U = 0, identity start).
template <typename TIn, int D, bool PERDIM>
__global__ void __launch_bounds__(NT, 1)
simt_pre_kernel(const cpdr_fragment *__restrict__ frags, const int32_t *__restrict__ items,
                const TIn *__restrict__ k, const TIn *__restrict__ v, const TIn *__restrict__ beta,
                const float *__restrict__ g, float *__restrict__ S_ext, float *__restrict__ M, int H,
                bool vfirst) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(smem_raw);
    constexpr int LB = Smem<D>::LB;
    const cpdr_fragment f = frags[items[blockIdx.x]];
    const int h = blockIdx.y;
    const bool mcols = blockIdx.z >= D / BV;
    const int col0 = (mcols ? blockIdx.z - D / BV : blockIdx.z) * BV;
    for (int idx = threadIdx.x; idx < D * BV; idx += NT) {
        const int d = idx / BV, c = idx % BV;
        s.S[d * LB + c] = (mcols && d == col0 + c) ? 1.f : 0.f;
    }
    for (int c0 = 0; c0 < f.len; c0 += C) {
        const int n = min(C, f.len - c0);
        const int64_t t0 = f.tok0 + c0;
        __syncthreads();
        load_chunk<TIn, D, PERDIM>(s, nullptr, k, beta, g, t0, n, H, h, H, h);
        build_A_QK<D, PERDIM, false>(s);
        __syncthreads();
        solve_WU<TIn, D, PERDIM>(s, v, t0, n, H, h, col0, mcols);
        __syncthreads();
        delta_step<D>(s);
        __syncthreads();
        state_step<D, PERDIM>(s, n);
    }
    __syncthreads();
    // M keeps [dk][dk]; S_ext follows the state layout
    float *dst = mcols ? M : S_ext;
    const bool vf = vfirst && !mcols;
    for (int idx = threadIdx.x; idx < D * BV; idx += NT) {
        const int d = vf ? idx % D : idx / BV, c = vf ? idx / D : idx % BV;
        dst[((int64_t)f.seg * H + h) * D * D + st_off<D>(d, col0 + c, vf)] = s.S[d * LB + c];
    }
}

// Merge: grid (chains, H, D / MBV).  S = S_ext[r0]; then for j = r0+1 .. r1-1:
// S <- M_j S + S_ext[j]; S_init[j] written after each step (S_init[r0+1] = S_ext[r0]).
// The CTA's (D x MBV) state tile stays in shared memory; M_j is staged
// row-major with cp.async, MNBUF - 1 steps ahead.  The K = D sum of a step is
// split over the four quarters of the CTA: a thread accumulates a (D/32 x 4)
// register tile (rows rb + 32a, columns 4cb ..) over its quarter of K, so
// that every value it loads from shared memory feeds four products; quarters
// 1-3 pass their partial sums through shared memory to quarter 0, which adds
// S_ext[j] and writes the new state.  The S_ext[j] tile is staged with M_j.
constexpr int MBV = 16;
constexpr int MNBUF = 2;
constexpr int MT = 512;        // merge threads: four quarters of 128

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N committed groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// VF: S_ext and S_init in the state_v_first layout [dv][dk]; the tile stays
// (key dim x value dim) in shared memory and only the global accesses turn.
template <int D, bool VF>
__global__ void __launch_bounds__(MT, 1)
merge_kernel(const MergeChain *__restrict__ chains, const float *__restrict__ S_ext,
             const float *__restrict__ M, float *__restrict__ S_init, int H, int B) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int LM = D + 4;                                  // padded row stride (16-byte rows)
    constexpr int RT = D / 32;                                 // rows per thread
    constexpr int KQ = D / 4;                                  // K per quarter of the CTA
    constexpr int NQ = MT / 4;                                 // threads per quarter
    float *Mn = reinterpret_cast<float *>(smem_raw);           // [MNBUF][D][LM]
    float *Ss = Mn + MNBUF * D * LM;                           // [D][MBV]
    float *Red = Ss + D * MBV;                                 // [3][RT][NQ][4] partial sums of quarters 1-3
    float *En = Red + 3 * RT * NQ * 4;                         // [MNBUF][D * MBV] S_ext tiles ([D][MBV]; VF: [MBV][D])
    const MergeChain ch = chains[blockIdx.x];
    const int h = blockIdx.y, col0 = blockIdx.z * MBV;
    auto idx_of = [&](int r) { return ((int64_t)(r * B + ch.b) * H + h) * D * D; };
    // stage M_j and the S_ext[j] tile into buffer (j - r0 - 1) % MNBUF (one
    // commit group per step, empty past the end)
    auto stage_M = [&](int j) {
        if (j < ch.r1) {
            const int bi = (j - ch.r0 - 1) % MNBUF;
            const float *Mj = M + idx_of(j);
            float *dst = Mn + bi * D * LM;
            for (int idx = threadIdx.x; idx < D * D / 4; idx += MT) {
                const int d = idx / (D / 4), l4 = idx % (D / 4);
                cp_async16(dst + d * LM + 4 * l4, Mj + d * D + 4 * l4);
            }
            const float *Ej = S_ext + idx_of(j);
            float *edst = En + bi * D * MBV;
            if (threadIdx.x < D * MBV / 4) {
                if (VF) {   // columns col0 .. col0 + MBV - 1 are whole rows of [dv][dk]
                    const int c = threadIdx.x / (D / 4), d4 = threadIdx.x % (D / 4);
                    cp_async16(edst + c * D + 4 * d4, Ej + (int64_t)(col0 + c) * D + 4 * d4);
                } else {
                    const int d = threadIdx.x / (MBV / 4), c4 = threadIdx.x % (MBV / 4);
                    cp_async16(edst + d * MBV + 4 * c4, Ej + (int64_t)d * D + col0 + 4 * c4);
                }
            }
        }
        cp_async_commit();
    };
    for (int idx = threadIdx.x; idx < D * MBV; idx += MT) {
        const int d = VF ? idx % D : idx / MBV, c = VF ? idx / D : idx % MBV;
        const int64_t off = st_off<D>(d, col0 + c, VF);
        const float x = S_ext[idx_of(ch.r0) + off];
        Ss[d * MBV + c] = x;
        S_init[idx_of(ch.r0 + 1) + off] = x;
    }
#pragma unroll
    for (int k = 1; k < MNBUF; k++) stage_M(ch.r0 + k);
    const int kh = threadIdx.x / NQ, u = threadIdx.x % NQ;
    const int rb = u >> 2, cb = (u & 3) * 4;
    for (int j = ch.r0 + 1; j < ch.r1; j++) {
        const int buf = (j - ch.r0 - 1) % MNBUF;
        cp_async_wait<MNBUF - 2>();
        __syncthreads();   // M_j staged; the previous step's state tile written
        stage_M(j + MNBUF - 1);
        const float *Mb = Mn + buf * D * LM;
        const float *Eb = En + buf * D * MBV;
        float acc[RT][4];
#pragma unroll
        for (int a = 0; a < RT; a++) {
            const int d = rb + 32 * a;
            float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kh == 0)
                e = VF ? make_float4(Eb[cb * D + d], Eb[(cb + 1) * D + d], Eb[(cb + 2) * D + d], Eb[(cb + 3) * D + d])
                       : *reinterpret_cast<const float4 *>(Eb + d * MBV + cb);
            acc[a][0] = e.x; acc[a][1] = e.y; acc[a][2] = e.z; acc[a][3] = e.w;
        }
        const int l0 = kh * KQ;
#pragma unroll 2
        for (int l = l0; l < l0 + KQ; l += 4) {
            float4 sv[4];
#pragma unroll
            for (int e = 0; e < 4; e++) sv[e] = *reinterpret_cast<const float4 *>(Ss + (l + e) * MBV + cb);
#pragma unroll
            for (int a = 0; a < RT; a++) {
                const float4 m = *reinterpret_cast<const float4 *>(Mb + (rb + 32 * a) * LM + l);
                const float mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    acc[a][0] = fmaf(mv[e], sv[e].x, acc[a][0]);
                    acc[a][1] = fmaf(mv[e], sv[e].y, acc[a][1]);
                    acc[a][2] = fmaf(mv[e], sv[e].z, acc[a][2]);
                    acc[a][3] = fmaf(mv[e], sv[e].w, acc[a][3]);
                }
            }
        }
        if (kh > 0) {
#pragma unroll
            for (int a = 0; a < RT; a++)
                *reinterpret_cast<float4 *>(Red + (((kh - 1) * RT + a) * NQ + u) * 4) =
                    make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
        __syncthreads();   // partial sums written; every thread has read the old state tile
        if (kh == 0) {
            float *dst = S_init + idx_of(j + 1);
#pragma unroll
            for (int a = 0; a < RT; a++) {
                float4 o = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
#pragma unroll
                for (int q = 0; q < 3; q++) {
                    const float4 pr = *reinterpret_cast<const float4 *>(Red + ((q * RT + a) * NQ + u) * 4);
                    o.x += pr.x; o.y += pr.y; o.z += pr.z; o.w += pr.w;
                }
                const int d = rb + 32 * a;
                *reinterpret_cast<float4 *>(Ss + d * MBV + cb) = o;
                if (VF) {
                    dst[st_off<D>(d, col0 + cb, true)] = o.x;
                    dst[st_off<D>(d, col0 + cb + 1, true)] = o.y;
                    dst[st_off<D>(d, col0 + cb + 2, true)] = o.z;
                    dst[st_off<D>(d, col0 + cb + 3, true)] = o.w;
                } else {
                    *reinterpret_cast<float4 *>(dst + d * D + col0 + cb) = o;
                }
            }
        }
    }
    cp_async_wait<0>();
}

// Zero [H, rows, width] slabs of the listed entries of a [*, H, rows, width] buffer.
__global__ void zero_slabs_kernel(const int32_t *__restrict__ list, float *__restrict__ buf,
                                  int64_t slab) {
    float4 *p = reinterpret_cast<float4 *>(buf + (int64_t)list[blockIdx.x] * slab);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = threadIdx.x + (int64_t)blockIdx.y * blockDim.x; i < slab / 4;
         i += (int64_t)blockDim.x * gridDim.y)
        p[i] = z;
}

template <typename TIn, int D, bool PERDIM>
int launch_fwd_t(const cpdr_ctx *c, const int32_t *items, int n_items, const void *q, const void *k, const void *v,
                 const void *beta, const float *g, const float *S_init, void *o, float *fs, cudaStream_t st) {
    const auto &p = c->plan;
    auto kern = simt_fwd_kernel<TIn, D, PERDIM>;
    const size_t sm = smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((unsigned)n_items, (unsigned)p.Hq, (unsigned)(D / BV));
    kern<<<grid, NT, sm, st>>>(c->dev.frags, items, (const TIn *)q, (const TIn *)k,
                               (const TIn *)v, (const TIn *)beta, g, S_init, (TIn *)o, fs, p.H, p.G,
                               p.vfirst, p.scale);
    return (int)cudaGetLastError();
}

template <typename TIn, int D, bool PERDIM>
int launch_pre_t(const cpdr_ctx *c, const void *k, const void *v, const void *beta, const float *g,
                 float *S_ext, float *M, cudaStream_t st) {
    const auto &p = c->plan;
    if (p.pre_items.empty()) return 0;
    auto kern = simt_pre_kernel<TIn, D, PERDIM>;
    const size_t sm = smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((unsigned)p.pre_items.size(), (unsigned)p.H, (unsigned)(2 * D / BV));
    kern<<<grid, NT, sm, st>>>(c->dev.frags, c->dev.pre_items, (const TIn *)k, (const TIn *)v,
                               (const TIn *)beta, g, S_ext, M, p.H, p.vfirst);
    return (int)cudaGetLastError();
}

template <typename TIn, int D>
int dispatch_gate_fwd(const cpdr_ctx *c, const int32_t *it, int n, const void *q, const void *k, const void *v,
                      const void *b, const float *g, const float *Si, void *o, float *fs, cudaStream_t st) {
    return c->plan.gate_kind == CPDR_GATE_PER_DIM
               ? launch_fwd_t<TIn, D, true>(c, it, n, q, k, v, b, g, Si, o, fs, st)
               : launch_fwd_t<TIn, D, false>(c, it, n, q, k, v, b, g, Si, o, fs, st);
}
template <typename TIn, int D>
int dispatch_gate_pre(const cpdr_ctx *c, const void *k, const void *v, const void *b, const float *g,
                      float *Se, float *M, cudaStream_t st) {
    return c->plan.gate_kind == CPDR_GATE_PER_DIM ? launch_pre_t<TIn, D, true>(c, k, v, b, g, Se, M, st)
                                                  : launch_pre_t<TIn, D, false>(c, k, v, b, g, Se, M, st);
}

}  // namespace

int launch_simt_fwd(const cpdr_ctx *c, const int32_t *items, int n, const void *q, const void *k, const void *v,
                    const void *beta, const float *g, const float *S_init, void *o, float *fs, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const auto &p = c->plan;
    if (n <= 0) return 0;
    if (p.in_dtype == CPDR_DTYPE_F32)
        return p.dk == 64 ? dispatch_gate_fwd<float, 64>(c, items, n, q, k, v, beta, g, S_init, o, fs, st)
                          : dispatch_gate_fwd<float, 128>(c, items, n, q, k, v, beta, g, S_init, o, fs, st);
    return p.dk == 64 ? dispatch_gate_fwd<__nv_bfloat16, 64>(c, items, n, q, k, v, beta, g, S_init, o, fs, st)
                      : dispatch_gate_fwd<__nv_bfloat16, 128>(c, items, n, q, k, v, beta, g, S_init, o, fs, st);
}

int launch_simt_pre(const cpdr_ctx *c, const void *k, const void *v, const void *beta, const float *g,
                    float *S_ext, float *M, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const auto &p = c->plan;
    if (p.in_dtype == CPDR_DTYPE_F32)
        return p.dk == 64 ? dispatch_gate_pre<float, 64>(c, k, v, beta, g, S_ext, M, st)
                          : dispatch_gate_pre<float, 128>(c, k, v, beta, g, S_ext, M, st);
    return p.dk == 64 ? dispatch_gate_pre<__nv_bfloat16, 64>(c, k, v, beta, g, S_ext, M, st)
                      : dispatch_gate_pre<__nv_bfloat16, 128>(c, k, v, beta, g, S_ext, M, st);
}

template <int D, bool VF>
int launch_merge_t(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init, cudaStream_t st) {
    const auto &p = c->plan;
    dim3 grid((unsigned)p.chains.size(), (unsigned)p.H, (unsigned)(D / MBV));
    const size_t sm = sizeof(float) * (MNBUF * D * (D + 4) + D * MBV + 3 * (D / 32) * MT + MNBUF * D * MBV);
    cudaError_t e = cudaFuncSetAttribute(merge_kernel<D, VF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return (int)e;
    merge_kernel<D, VF><<<grid, MT, sm, st>>>(c->dev.chains, S_ext, M, S_init, p.H, p.B);
    return (int)cudaGetLastError();
}

int launch_merge(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const auto &p = c->plan;
    if (p.chains.empty()) return 0;
    if (c->use_tc && p.dk == 128) return launch_tc_merge(c, S_ext, M, S_init, stream);
    if (p.dk == 64)
        return p.vfirst ? launch_merge_t<64, true>(c, S_ext, M, S_init, st)
                        : launch_merge_t<64, false>(c, S_ext, M, S_init, st);
    return p.vfirst ? launch_merge_t<128, true>(c, S_ext, M, S_init, st)
                    : launch_merge_t<128, false>(c, S_ext, M, S_init, st);
}

int launches_per_step(const cpdr_ctx *c) {
    const auto &p = c->plan;
    int n = 0;
    // WY build (tensor-core path; the per-dim gate's preparation and solve)
    n += (c->use_tc && !p.wy_chunks.empty()) ? (p.gate_kind == CPDR_GATE_PER_DIM ? 2 : 1) : 0;
    n += p.pre_items.empty() ? 0 : 1;          // pre-process (S and M chains in one launch on the tensor cores)
    n += p.zero_pre.empty() ? 0 : 2;           // zero S_ext and M
    n += p.zero_init.empty() ? 0 : 1;          // zero S_init
    n += p.chains.empty() ? 0 : 1;             // merge
    n += p.frags.empty() ? 0 : 1;              // forward
    n += p.empty_seqs.empty() ? 0 : 1;         // zero final states of empty sequences
    return n;
}

// which: 0 = S_ext and M of zero_pre, 1 = S_init of zero_init, 2 = final states of empty sequences
int launch_zero_segments(const cpdr_ctx *c, float *S_ext, float *M, float *S_init, float *fs, int which,
                         void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const auto &p = c->plan;
    const int64_t slab_s = (int64_t)p.H * p.dk * p.dv, slab_m = (int64_t)p.H * p.dk * p.dk;
    const dim3 blk(256);
    if (which == 0 && !p.zero_pre.empty()) {
        dim3 grid((unsigned)p.zero_pre.size(), 8);
        zero_slabs_kernel<<<grid, blk, 0, st>>>(c->dev.zero_pre, S_ext, slab_s);
        zero_slabs_kernel<<<grid, blk, 0, st>>>(c->dev.zero_pre, M, slab_m);
    } else if (which == 1 && !p.zero_init.empty()) {
        dim3 grid((unsigned)p.zero_init.size(), 8);
        zero_slabs_kernel<<<grid, blk, 0, st>>>(c->dev.zero_init, S_init, slab_s);
    } else if (which == 2 && !p.empty_seqs.empty() && fs) {
        dim3 grid((unsigned)p.empty_seqs.size(), 8);
        zero_slabs_kernel<<<grid, blk, 0, st>>>(c->dev.empty_seqs, fs, slab_s);
    }
    return (int)cudaGetLastError();
}

}  // namespace cpdr
