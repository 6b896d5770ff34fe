// Tensor-core merge for the bf16, d = 128 path: along each sequence chain
// r0 < r1 of one row b ([FLA-CP] §2.1 merge, §5.2)
//   S = S_ext[r0];  S_init[r0+1] = S
//   for j = r0+1 .. r1-1:  S <- M_j S + S_ext[j];  S_init[j+1] = S
// as tcgen05 products D = M_j S with fp32 accumulation in TMEM.  M_j and S
// enter the tensor core as bf16 hi/lo pairs (x = hi + lo, hi = bf16(x),
// lo = bf16(x - hi)), D = hi(M) hi(S) + lo(M) hi(S) + hi(M) lo(S), the same
// split the transfer-matrix chain uses, so the scan keeps close to fp32
// accuracy (the dropped lo*lo term is below 2^-16 relative).
//
// CTA = (chain, head, 16 or 32 state columns): 13 warps.  Warps 5-12 convert M_j
// (fp32, row-major [dk][dk] = K-major A; 16 rows per warp, each read as one
// coalesced 512-byte row) into the two bf16 images of a double buffer, one
// step ahead; warp 4 issues the three products per step
// (M = 128, N = 16 or 32, K = 128); warps 0-3 own state rows 32w .. 32w + 31 (their
// TMEM lane quarter): they read D, add S_ext[j], write the new state's hi/lo
// images as the next B operand (K-major: B^T[n][k] = S[k][n]) and S_init[j+1].
// Every wait is bounded as in the chain kernels.
//
// The same kernel runs the backward's reverse merge (rev = 1): along each
// chain, from its last segment down,
//   G = dS_ext[r1];  dS_end[r1-1] = G
//   for j = r1-1 .. r0+1:  G <- M_j^T G + dS_ext[j];  dS_end[j-1] = G
// with the transposed transfer matrices of the article's backward (§2.2).
// M_j's bf16 image is the same; the products read it as an MN-major A
// operand, which is M_j^T.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"

namespace cpdr {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int kEpiWarps = 4;                     // warps 0-3: state rows
constexpr int kMmaWarp = 4;                      // warp 4: products, TMEM owner
constexpr int kCvtWarps = 8;                     // warps 5-12: M_j to bf16 hi/lo
constexpr int kThreads = 32 * (kEpiWarps + 1 + kCvtWarps);
constexpr uint32_t kTmemCols = 32;

// Shared memory (offsets from a 1024-aligned base).  A image: 128 x 128 bf16,
// K-major with 128-byte swizzle, two 64-column atoms of 16 KiB; B image:
// B^T (NB x 128), two atoms of NB x 128 bytes.
constexpr uint32_t kATile = D * D * 2;
constexpr uint32_t kAAtom = D * 128;
constexpr uint32_t O_A = 0;                      // [buffer 0, 1][hi, lo]
constexpr uint32_t O_B = 4 * kATile;             // [hi, lo]
enum MergeBar { MB_AFULL0, MB_AFULL1, MB_AFREE0, MB_AFREE1, MB_BFULL, MB_DFULL, MB_DRAIN, MB_N };
static_assert(MB_N * 8 <= 64, "merge barriers exceed their slot");
template <int NB>
struct MLay {
    static_assert(NB == 16 || NB == 32, "state columns per CTA");
    static constexpr uint32_t kBTile = NB * D * 2;
    static constexpr uint32_t kBAtom = NB * 128;
    static constexpr int kXS = NB + 4;                  // row stride (floats) of the transpose scratch
    static constexpr uint32_t O_X = O_B + 2 * kBTile;   // per state-row warp: 32 x kXS floats
    static constexpr uint32_t O_BARS = O_X + kEpiWarps * 32 * kXS * 4;
    static constexpr uint32_t O_CTL = O_BARS + 64;
    static constexpr uint32_t O_TSLOT = O_CTL + 16;
    static constexpr uint32_t kSmem = O_TSLOT + 16;
    static_assert(kSmem + 1024 <= 232448, "merge layout exceeds shared memory");
};

struct MergeArgs {
    const MergeChain *chains;
    const float *S_ext;
    const float *M;
    float *S_init;
    int32_t *status;
    int H, B, vfirst;
    int rev;          // 1: the reverse merge (M_j^T, chain walked from r1 down)
};

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, Ctl *ctl, int32_t *status, int site) {
    return warp_wait_all(bar, parity, ctl, status, site);
}

// bf16 hi/lo of two values, packed (lower column in the low half)
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(a, b);
    const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
    lo = pack_bf16(a - h.x, b - h.y);
}

// NB: state columns per CTA (the products' N), 16 or 32
template <int NB>
__global__ void __launch_bounds__(kThreads, 1) tc_merge_kernel(const __grid_constant__ MergeArgs p) {
    using L = MLay<NB>;
    constexpr uint32_t kBTile = L::kBTile, kBAtom = L::kBAtom, O_X = L::O_X, O_BARS = L::O_BARS, O_CTL = L::O_CTL,
                       O_TSLOT = L::O_TSLOT;
    constexpr int kXS = L::kXS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + O_BARS);
    Ctl *ctl = reinterpret_cast<Ctl *>(base + O_CTL);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + O_TSLOT);
    const MergeChain ch = p.chains[blockIdx.x];
    const int h = blockIdx.y, col0 = blockIdx.z * NB;
    const int nsteps = ch.r1 - ch.r0 - 1;   // steps j = r0+1 .. r1-1 (reverse: r1-1 .. r0+1)
    auto idx_of = [&](int r) { return ((int64_t)(r * p.B + ch.b) * p.H + h) * D * D; };
    const bool rev = p.rev != 0;
    const int first = rev ? ch.r1 : ch.r0;                                       // segment of the first S_ext
    auto jstep = [&](int step) { return rev ? ch.r1 - 1 - step : ch.r0 + 1 + step; };
    auto out_of = [&](int j) { return rev ? j - 1 : j + 1; };                    // segment written after j

    if (threadIdx.x == 0) {
        mbar_init(&bar[MB_AFULL0], kCvtWarps);
        mbar_init(&bar[MB_AFULL1], kCvtWarps);
        mbar_init(&bar[MB_AFREE0], 1);
        mbar_init(&bar[MB_AFREE1], 1);
        mbar_init(&bar[MB_BFULL], kEpiWarps);
        mbar_init(&bar[MB_DFULL], 1);
        mbar_init(&bar[MB_DRAIN], 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == kMmaWarp) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (w < kEpiWarps) {
        // ------------------------------------------------------------ state rows
        const int d = 32 * w + lane;
        uint8_t *bhi = base + O_B, *blo = base + O_B + kBTile;
        // element (n, d) of B^T: atom d / 64, 16-byte chunk (d % 64) / 8
        const uint32_t boff = (uint32_t)(d >> 6) * kBAtom + (uint32_t)((d & 7) * 2);
        const uint32_t bchunk = (uint32_t)((d & 63) >> 3);
        // global rows of the tile (row d: NB floats): [dv][dk] states are
        // column-major per thread, so lanes read consecutive floats; [dk][dv]
        // rows go through a per-warp scratch so that a warp moves whole
        // rows per access instead of 32 separate pieces
        float *xs = reinterpret_cast<float *>(base + O_X) + w * 32 * kXS;
        // coalesced side: NB / 4 lanes per row, 128 / NB rows per access
        constexpr int kLPR = NB / 4, kRPI = 32 / kLPR;
        const int xr = lane / kLPR, xq = lane % kLPR;
        auto load_row = [&](const float *src, float (&x)[NB]) {
            if (p.vfirst) {
#pragma unroll
                for (int n = 0; n < NB; n++) x[n] = src[(int64_t)(col0 + n) * D + d];
            } else {
                const float *g = src + (int64_t)(32 * w) * D + col0;
#pragma unroll
                for (int i = 0; i < kLPR; i++) {
                    const int r = xr + kRPI * i;
                    *reinterpret_cast<float4 *>(xs + r * kXS + 4 * xq) =
                        *reinterpret_cast<const float4 *>(g + (int64_t)r * D + 4 * xq);
                }
                __syncwarp();
#pragma unroll
                for (int n4 = 0; n4 < NB / 4; n4++) {
                    const float4 v = *reinterpret_cast<const float4 *>(xs + lane * kXS + 4 * n4);
                    x[4 * n4] = v.x; x[4 * n4 + 1] = v.y; x[4 * n4 + 2] = v.z; x[4 * n4 + 3] = v.w;
                }
                __syncwarp();
            }
        };
        auto store_row = [&](float *dst, const float (&x)[NB]) {
            if (p.vfirst) {
#pragma unroll
                for (int n = 0; n < NB; n++) dst[(int64_t)(col0 + n) * D + d] = x[n];
            } else {
#pragma unroll
                for (int n4 = 0; n4 < NB / 4; n4++)
                    *reinterpret_cast<float4 *>(xs + lane * kXS + 4 * n4) =
                        make_float4(x[4 * n4], x[4 * n4 + 1], x[4 * n4 + 2], x[4 * n4 + 3]);
                __syncwarp();
                float *g = dst + (int64_t)(32 * w) * D + col0;
#pragma unroll
                for (int i = 0; i < kLPR; i++) {
                    const int r = xr + kRPI * i;
                    *reinterpret_cast<float4 *>(g + (int64_t)r * D + 4 * xq) =
                        *reinterpret_cast<const float4 *>(xs + r * kXS + 4 * xq);
                }
                __syncwarp();
            }
        };
        // the state's hi/lo images as the next B operand (this thread: column d of B^T)
        auto put_b = [&](const float (&x)[NB]) {
#pragma unroll
            for (int n = 0; n < NB; n += 2) {
                uint32_t hi, lo;
                split2(x[n], x[n + 1], hi, lo);
                const uint32_t o0 = boff + sw128((uint32_t)n, bchunk), o1 = boff + sw128((uint32_t)n + 1, bchunk);
                *reinterpret_cast<uint16_t *>(bhi + o0) = (uint16_t)(hi & 0xffffu);
                *reinterpret_cast<uint16_t *>(bhi + o1) = (uint16_t)(hi >> 16);
                *reinterpret_cast<uint16_t *>(blo + o0) = (uint16_t)(lo & 0xffffu);
                *reinterpret_cast<uint16_t *>(blo + o1) = (uint16_t)(lo >> 16);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[MB_BFULL]);
        };
        float s[NB], e[NB];
        load_row(p.S_ext + idx_of(first), s);
        store_row(p.S_init + idx_of(out_of(first)), s);
        if (nsteps > 0) {
            put_b(s);
            load_row(p.S_ext + idx_of(jstep(0)), e);
        }
        for (int step = 0; step < nsteps; step++) {
            const int j = jstep(step);
            if (!warp_wait_bar(&bar[MB_DFULL], step & 1, ctl, p.status, 130)) break;
            tc_fence_after();
            float v[32];
            if (NB == 32) tmem_ld32(tmem + ((uint32_t)(32 * w) << 16), v);
            else tmem_ld16(tmem + ((uint32_t)(32 * w) << 16), reinterpret_cast<float (&)[16]>(v));
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < NB; n++) s[n] = v[n] + e[n];
            tc_fence_before();
            if (step + 1 < nsteps) put_b(s);   // the next product may start
            store_row(p.S_init + idx_of(out_of(j)), s);
            if (step + 1 < nsteps) load_row(p.S_ext + idx_of(jstep(step + 1)), e);
        }
    } else if (w == kMmaWarp) {
        // ------------------------------------------------------------ products
        if (lane == 0) {
            // A = M_j (K-major image) or, reverse, M_j^T (the same image read MN-major)
            const uint32_t id = rev ? idesc_bf16(128, NB, true, false) : idesc_bf16(128, NB, false, false);
            const uint32_t a0 = smem_u32(base + O_A), b0 = smem_u32(base + O_B);
            for (int step = 0; step < nsteps; step++) {
                const int buf = step & 1;
                if (!mbar_wait(&bar[MB_AFULL0 + buf], (step >> 1) & 1, ctl, p.status, 131)) break;
                if (!mbar_wait(&bar[MB_BFULL], step & 1, ctl, p.status, 132)) break;
                tc_fence_after();
                const uint32_t ahi = a0 + (uint32_t)(2 * buf) * kATile, alo = ahi + kATile;
                const uint32_t bhi = b0, blo = b0 + kBTile;
                // D = hi(M) hi(S) + lo(M) hi(S) + hi(M) lo(S)
                const uint32_t as[3] = {ahi, alo, ahi}, bs[3] = {bhi, bhi, blo};
#pragma unroll
                for (int t = 0; t < 3; t++) {
                    // K-major: 128-byte swizzle, K atoms kAAtom apart; MN-major: M atoms
                    // kAAtom apart (LBO), 16 K rows per step
                    const uint64_t ad = rev ? sdesc(as[t], kAAtom, 1024) : sdesc(as[t], 16, 1024);
                    const uint64_t bd = sdesc(bs[t], 16, 1024);
#pragma unroll
                    for (int k = 0; k < D / 16; k++) {
                        const uint64_t ao = rev ? (uint64_t)(k * 128) : ((k & 3) * 32 + (k >> 2) * kAAtom) >> 4;
                        const uint64_t bo = ((k & 3) * 32 + (k >> 2) * kBAtom) >> 4;
                        mma_bf16(tmem, ad + ao, bd + bo, id, (t > 0 || k > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&bar[MB_AFREE0 + buf]);
                mma_commit(&bar[MB_DFULL]);
            }
            mma_commit(&bar[MB_DRAIN]);
            Ctl local;
            local.abort = 0;
            mbar_wait(&bar[MB_DRAIN], 0, &local, p.status, 133);
        }
    } else {
        // ------------------------------------------------------------ M_j to bf16 hi/lo
        // converter warp cw: rows 16 cw .. 16 cw + 15 of M_j, lane l holding
        // columns 4l .. 4l + 3 of each (one coalesced 512-byte row per load);
        // the next step's rows are loaded as soon as this step's are stored
        const int cw = w - (kEpiWarps + 1);
        const uint32_t aoff = (uint32_t)(lane >> 4) * kAAtom + (uint32_t)(lane & 1) * 8;
        const uint32_t achunk = (uint32_t)((lane & 15) >> 1);
        float4 x[16];
        auto load_m = [&](int step) {
            const float4 *src = reinterpret_cast<const float4 *>(p.M + idx_of(jstep(step))) + (16 * cw) * (D / 4) + lane;
#pragma unroll
            for (int i = 0; i < 16; i++) x[i] = src[i * (D / 4)];
        };
        if (nsteps > 0) load_m(0);
        for (int step = 0; step < nsteps; step++) {
            const int buf = step & 1;
            if (step >= 2 && !warp_wait_bar(&bar[MB_AFREE0 + buf], ((step - 2) >> 1) & 1, ctl, p.status, 134)) break;
            uint8_t *hi = base + O_A + (uint32_t)(2 * buf) * kATile + aoff;
            uint8_t *lo = hi + kATile;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                uint32_t h0, l0, h1, l1;
                split2(x[i].x, x[i].y, h0, l0);
                split2(x[i].z, x[i].w, h1, l1);
                const uint32_t o = sw128((uint32_t)(16 * cw + i), achunk);
                *reinterpret_cast<uint2 *>(hi + o) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(lo + o) = make_uint2(l0, l1);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[MB_AFULL0 + buf]);
            if (step + 1 < nsteps) load_m(step + 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {
int launch_merge_dir(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init, int rev, void *stream) {
    const auto &pl = c->plan;
    if (pl.chains.empty()) return 0;
    MergeArgs a{};
    a.chains = c->dev.chains;
    a.S_ext = S_ext;
    a.M = M;
    a.S_init = S_init;
    a.status = c->dev.status;
    a.H = pl.H;
    a.B = pl.B;
    a.vfirst = (pl.vfirst && !rev) ? 1 : 0;
    a.rev = rev;
    // 16-column tiles while they fit one wave (one CTA per SM), else 32
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int64_t ctas16 = (int64_t)pl.chains.size() * pl.H * (D / 16);
    auto go = [&](auto kern, int nb, size_t smem) -> int {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        dim3 grid((unsigned)pl.chains.size(), (unsigned)pl.H, (unsigned)(D / nb));
        kern<<<grid, kThreads, smem, (cudaStream_t)stream>>>(a);
        return (int)cudaGetLastError();
    };
    if (ctas16 <= sms) return go(tc_merge_kernel<16>, 16, MLay<16>::kSmem + 1024);
    return go(tc_merge_kernel<32>, 32, MLay<32>::kSmem + 1024);
}
}  // namespace

int launch_tc_merge(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init, void *stream) {
    return launch_merge_dir(c, S_ext, M, S_init, 0, stream);
}

// The backward's reverse merge: dS_end from dS_ext and M ([dk][dv] states).
int launch_tc_merge_rev(const cpdr_ctx *c, const float *dS_ext, const float *M, float *dS_end, void *stream) {
    return launch_merge_dir(c, dS_ext, M, dS_end, 1, stream);
}

}  // namespace cpdr
