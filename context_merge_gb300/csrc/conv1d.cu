// Causal depthwise conv1d on the context's segments: the layer step before
// the delta rule.  The article "flash-linear-attention 上下文并行CP ..."
// ([FLA-CP]) gives its context-parallel form: the conv reaches W - 1 tokens
// back, so a rank needs the tail of the previous rank's tokens (§2.4,
// send_recv_fwd) and the context records how many of them belong to its
// first sequence (§3.3, pre_num_conv_tokens).  On one device the tail is read
// where it lies in memory -- right before the tile, or, for a segment's first
// tile, at the positions the planner's halo table lists (another part of the
// zigzag layout, or earlier parts when parts are shorter than W - 1).
//
// HBM-bound streaming kernel: each thread owns 2 channels (4 bytes of bf16,
// 8 of fp32) of one tile of up to 64 tokens, keeps the W - 1 previous inputs
// in registers, and reads each input and writes each output once.  Loads go
// out in groups of 16 tokens, the next group before the current one is used;
// few registers per thread keep the SM full of warps (the loads in flight
// are what bounds a streaming kernel).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"

namespace cpdr {
namespace {

constexpr int kConvThreads = 256;
constexpr int kVec = 2;          // channels per thread
constexpr int kAhead = 16;       // tokens per load group (two groups in flight)

struct Vec2 {
    float v[kVec];
};

// 2 channels as loaded (raw bits), widened to fp32 where they are used
template <typename T>
struct Raw2;
template <>
struct Raw2<float> {
    float2 a;
};
template <>
struct Raw2<__nv_bfloat16> {
    uint32_t a;
};

__device__ __forceinline__ Raw2<float> load_raw(const float *p) {
    return Raw2<float>{__ldg(reinterpret_cast<const float2 *>(p))};
}
__device__ __forceinline__ Raw2<__nv_bfloat16> load_raw(const __nv_bfloat16 *p) {
    return Raw2<__nv_bfloat16>{__ldg(reinterpret_cast<const unsigned int *>(p))};
}
__device__ __forceinline__ Vec2 widen(const Raw2<float> &r) { return Vec2{{r.a.x, r.a.y}}; }
__device__ __forceinline__ Vec2 widen(const Raw2<__nv_bfloat16> &r) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.a));
    return Vec2{{f.x, f.y}};
}
template <typename T>
__device__ __forceinline__ Vec2 load2(const T *p) { return widen(load_raw(p)); }
__device__ __forceinline__ void store2(float *p, const Vec2 &x) {
    *reinterpret_cast<float2 *>(p) = make_float2(x.v[0], x.v[1]);
}
__device__ __forceinline__ void store2(__nv_bfloat16 *p, const Vec2 &x) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x.v[0], x.v[1]);
    *reinterpret_cast<__nv_bfloat162 *>(p) = h;
}

// SiLU z * sigmoid(z) = z / (1 + e^-z); the fast divide returns 0 once the
// denominator passes 2^126, where the exact quotient is below 1e-36
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// grid (conv tiles, channel blocks of kVec * kConvThreads)
template <typename T, int W, int ACT>
__global__ void __launch_bounds__(kConvThreads)
conv1d_kernel(const ConvTile *__restrict__ tiles, const int64_t *__restrict__ halo, const T *__restrict__ x,
              const float *__restrict__ weight, const float *__restrict__ bias, T *__restrict__ y, int channels) {
    const ConvTile tl = tiles[blockIdx.x];
    const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * kVec;
    if (c0 >= channels) return;
    const T *xp = x + tl.tok0 * channels + c0;
    T *yp = y + tl.tok0 * channels + c0;
    // first load group in flight before anything else
    Raw2<T> raw[2][kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; u++)
        if (u < tl.n) raw[0][u] = load_raw(xp + (int64_t)u * channels);
    float w[kVec][W], b[kVec];
#pragma unroll
    for (int j = 0; j < kVec; j++) {
#pragma unroll
        for (int i = 0; i < W; i++) w[j][i] = __ldg(weight + (int64_t)(c0 + j) * W + i);
        b[j] = bias ? __ldg(bias + c0 + j) : 0.f;
    }
    // the W - 1 inputs before the tile, oldest first
    constexpr int NW = W > 1 ? W - 1 : 1;
    Vec2 win[NW];
#pragma unroll
    for (int i = 0; i < NW; i++) {
        int64_t src = -1;
        if (W > 1) {
            if (tl.halo == kHaloMemory) src = tl.tok0 - (W - 1) + i;
            else if (tl.halo >= 0) src = __ldg(halo + (int64_t)tl.halo * (W - 1) + i);
        }
        if (src >= 0) win[i] = load2(x + src * channels + c0);
        else win[i] = Vec2{{0.f, 0.f}};
    }
    // groups of kAhead tokens; group g + 1 is loaded before group g is computed
#pragma unroll 1
    for (int t0 = 0; t0 < tl.n; t0 += 2 * kAhead) {
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const int g0 = t0 + half * kAhead;
            if (g0 >= tl.n) break;
            const int nxt = g0 + kAhead;
#pragma unroll
            for (int u = 0; u < kAhead; u++)
                if (nxt + u < tl.n) raw[half ^ 1][u] = load_raw(xp + (int64_t)(nxt + u) * channels);
#pragma unroll
            for (int u = 0; u < kAhead; u++) {
                if (g0 + u < tl.n) {
                    const Vec2 cur = widen(raw[half][u]);
                    Vec2 out;
#pragma unroll
                    for (int j = 0; j < kVec; j++) {
                        float acc = b[j];
#pragma unroll
                        for (int i = 0; i < W - 1; i++) acc = fmaf(w[j][i], win[i].v[j], acc);
                        acc = fmaf(w[j][W - 1], cur.v[j], acc);
                        out.v[j] = ACT ? silu(acc) : acc;
                    }
                    store2(yp + (int64_t)(g0 + u) * channels, out);
#pragma unroll
                    for (int i = 0; i + 1 < W - 1; i++) win[i] = win[i + 1];
                    if (W > 1) win[NW - 1] = cur;
                }
            }
        }
    }
}

template <typename T, int W>
int launch_w(const cpdr_ctx *c, const void *x, const float *weight, const float *bias, int channels, int act,
             void *y, cudaStream_t st) {
    const auto &p = c->plan;
    const dim3 grid((unsigned)p.conv_tiles.size(), (unsigned)((channels + kVec * kConvThreads - 1) /
                                                              (kVec * kConvThreads)));
    if (act)
        conv1d_kernel<T, W, 1><<<grid, kConvThreads, 0, st>>>(c->dev.conv_tiles, c->dev.conv_halo,
                                                               (const T *)x, weight, bias, (T *)y, channels);
    else
        conv1d_kernel<T, W, 0><<<grid, kConvThreads, 0, st>>>(c->dev.conv_tiles, c->dev.conv_halo,
                                                               (const T *)x, weight, bias, (T *)y, channels);
    return (int)cudaGetLastError();
}

template <typename T>
int launch_t(const cpdr_ctx *c, const void *x, const float *weight, const float *bias, int channels, int act,
             void *y, cudaStream_t st) {
    switch (c->plan.conv_width) {
        case 1: return launch_w<T, 1>(c, x, weight, bias, channels, act, y, st);
        case 2: return launch_w<T, 2>(c, x, weight, bias, channels, act, y, st);
        case 3: return launch_w<T, 3>(c, x, weight, bias, channels, act, y, st);
        case 4: return launch_w<T, 4>(c, x, weight, bias, channels, act, y, st);
        case 5: return launch_w<T, 5>(c, x, weight, bias, channels, act, y, st);
        case 6: return launch_w<T, 6>(c, x, weight, bias, channels, act, y, st);
        case 7: return launch_w<T, 7>(c, x, weight, bias, channels, act, y, st);
        case 8: return launch_w<T, 8>(c, x, weight, bias, channels, act, y, st);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace

static_assert(kMaxConvWidth == 8, "conv1d dispatch covers widths 1..8");

int launch_conv1d(const cpdr_ctx *c, const void *x, const float *weight, const float *bias, int channels,
                  int activation, void *y, void *stream) {
    if (c->plan.conv_tiles.empty()) return 0;
    cudaStream_t st = (cudaStream_t)stream;
    return c->plan.in_dtype == CPDR_DTYPE_F32
               ? launch_t<float>(c, x, weight, bias, channels, activation, y, st)
               : launch_t<__nv_bfloat16>(c, x, weight, bias, channels, activation, y, st);
}

}  // namespace cpdr
