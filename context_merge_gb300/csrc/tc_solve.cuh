// Solve of the per-chunk WY inverse T = (I + A)^-1 by a pair of warps per
// unit (the WY build of the scalar-gate path, tc_wy.cu, and the per-dim
// gate's solve kernel, tc_kda.cu).
#pragma once
#include <cuda_bf16.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"

namespace cpdr {
namespace tc {

constexpr int kLS = 68;   // row stride (floats) of the A scratch

// Converts T (rows in S[64][kLS], columns 0..63; the upper-right 32 x 32
// block is taken as zero whatever S holds there) into T' = T diag(beta) and
// T'' = T diag(beta gamma) (hi, lo), bf16, 16-byte pieces: lane l takes
// columns 8c .. 8c + 7 (c = l & 7) of rows 4p + r, p in [p0, p0 + np), with
// r = (l >> 3) ^ (c >> 2) so that the eight lanes of each quarter-warp read
// distinct bank groups; a warp stores four whole tile rows at a time.
__device__ __forceinline__ void store_tiles(const float *S, uint8_t *dst, const float *beta, const float *gam, int p0,
                                            int np) {
    const int l = threadIdx.x & 31;
    const int c = l & 7, r = (l >> 3) ^ (c >> 2);
    float bc[8], gc[8];
#pragma unroll
    for (int e = 0; e < 8; e++) {
        bc[e] = beta[8 * c + e];
        gc[e] = bc[e] * gam[8 * c + e];
    }
#pragma unroll 4
    for (int p = p0; p < p0 + np; p++) {
        const int i = 4 * p + r;
        float t[8];
        if (i < 32 && c >= 4) {
#pragma unroll
            for (int e = 0; e < 8; e++) t[e] = 0.f;
        } else {
            const float4 a0 = *reinterpret_cast<const float4 *>(S + i * kLS + 8 * c);
            const float4 a1 = *reinterpret_cast<const float4 *>(S + i * kLS + 8 * c + 4);
            t[0] = a0.x; t[1] = a0.y; t[2] = a0.z; t[3] = a0.w;
            t[4] = a1.x; t[5] = a1.y; t[6] = a1.z; t[7] = a1.w;
        }
        uint32_t u[4], hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            u[e] = pack_bf16(t[2 * e] * bc[2 * e], t[2 * e + 1] * bc[2 * e + 1]);
            const float w0 = t[2 * e] * gc[2 * e], w1 = t[2 * e + 1] * gc[2 * e + 1];
            hi[e] = pack_bf16(w0, w1);
            const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi[e]));
            lo[e] = pack_bf16(w0 - h.x, w1 - h.y);
        }
        const uint32_t o = sw128((uint32_t)i, (uint32_t)c);
        *reinterpret_cast<uint4 *>(dst + o) = make_uint4(u[0], u[1], u[2], u[3]);
        *reinterpret_cast<uint4 *>(dst + kWyTileBytes + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dst + 2 * kWyTileBytes + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Two warps (role 0 and 1, meeting at named barrier `bar_id`) solve one unit
// by blocks of the unit lower-triangular L = I + A, inverting blocks bottom
// up and forming every off-diagonal block as a product, which reuses each
// shared-memory value for several outputs (a forward substitution reads one
// broadcast value per product and runs out of shared-memory wavefronts):
//   16 x 16 diagonal blocks: forward substitution, T_i = e_i - sum_{k<i}
//       A_ik T_k, one block per half-warp, lane = column;
//   32 x 32 diagonal blocks (role r takes rows/cols 32r ..): with s, t its
//       two 16-blocks, T_ts = -T_tt (A_ts T_ss), 2 x 4 outputs per lane;
//   the 64 x 64 unit: T21 = -T22 (A21 T11), 4 x 4 outputs per lane over
//       both warps.
// T replaces A in S block by block; the products go through the upper-right
// 32 x 32 block of S, which A leaves unused (it is treated as zero after).
// Row sets are interleaved (rows rg, rg + 8, ...) so that the distinct rows
// a warp reads at once fall in distinct bank groups.
__device__ __forceinline__ void fma44(float (&x)[4][4], const float4 (&a)[4], const float4 (&b)[4]) {
#pragma unroll
    for (int r = 0; r < 4; r++) {
        const float av[4] = {a[r].x, a[r].y, a[r].z, a[r].w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            x[r][0] = fmaf(av[e], b[e].x, x[r][0]);
            x[r][1] = fmaf(av[e], b[e].y, x[r][1]);
            x[r][2] = fmaf(av[e], b[e].z, x[r][2]);
            x[r][3] = fmaf(av[e], b[e].w, x[r][3]);
        }
    }
}
__device__ __forceinline__ void fma24(float (&x)[2][4], const float4 (&a)[2], const float4 (&b)[4]) {
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const float av[4] = {a[r].x, a[r].y, a[r].z, a[r].w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            x[r][0] = fmaf(av[e], b[e].x, x[r][0]);
            x[r][1] = fmaf(av[e], b[e].y, x[r][1]);
            x[r][2] = fmaf(av[e], b[e].z, x[r][2]);
            x[r][3] = fmaf(av[e], b[e].w, x[r][3]);
        }
    }
}
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

// T itself as fp32 64 x 64 row-major (the upper-right 32 x 32 block, scratch
// during the solve, written as zero): role r of the pair writes rows
// 32 r .. 32 r + 31, the lanes across each row.
__device__ __forceinline__ void store_t_f32(const float *S, float *dst, int role) {
    const int l = threadIdx.x & 31;
#pragma unroll 4
    for (int rr = 0; rr < 32; rr++) {
        const int i = 32 * role + rr;
        dst[i * 64 + l] = S[i * kLS + l];
        dst[i * 64 + 32 + l] = i < 32 ? 0.f : S[i * kLS + 32 + l];
    }
}

__device__ __forceinline__ void solve_unit_pair(float *S, uint8_t *dst, const float *beta, const float *gam, int role,
                                                int bar_id, float *tdst = nullptr) {
    const int l = threadIdx.x & 31;
    const int o = 32 * role;
    {
        // 16 x 16 diagonal blocks o and o + 16, one per half-warp
        const int c = l & 15, b0 = o + 16 * (l >> 4);
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k4 = 0; k4 < 4; k4++) {
                if (4 * k4 >= i) break;
                const float4 v = ld4(S + (b0 + i) * kLS + b0 + 4 * k4);
                const float av[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; e++)
                    if (4 * k4 + e < i) a[e] = fmaf(av[e], y[4 * k4 + e], a[e]);
            }
            y[i] = (i == c ? 1.f : 0.f) - ((a[0] + a[1]) + (a[2] + a[3]));
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; i++) S[(b0 + i) * kLS + b0 + c] = y[i];
        __syncwarp();
    }
    {
        // this role's 32-block: X1 = A_ts T_ss into rows 16 role .. of the
        // upper-right block, then T_ts = -T_tt X1 over A_ts
        const int rg = l >> 2, cg = l & 3;
        const int s0 = o, t0 = o + 16, x0 = 16 * role;
        float x[2][4] = {};
#pragma unroll
        for (int k4 = 0; k4 < 4; k4++) {
            const float4 av[2] = {ld4(S + (t0 + rg) * kLS + s0 + 4 * k4), ld4(S + (t0 + rg + 8) * kLS + s0 + 4 * k4)};
            float4 bv[4];
#pragma unroll
            for (int e = 0; e < 4; e++) bv[e] = ld4(S + (s0 + 4 * k4 + e) * kLS + s0 + 4 * cg);
            fma24(x, av, bv);
        }
#pragma unroll
        for (int r = 0; r < 2; r++) st4(S + (x0 + rg + 8 * r) * kLS + 32 + 4 * cg, x[r][0], x[r][1], x[r][2], x[r][3]);
        __syncwarp();
        float z[2][4] = {};
#pragma unroll
        for (int k4 = 0; k4 < 4; k4++) {
            const float4 av[2] = {ld4(S + (t0 + rg) * kLS + t0 + 4 * k4), ld4(S + (t0 + rg + 8) * kLS + t0 + 4 * k4)};
            float4 bv[4];
#pragma unroll
            for (int e = 0; e < 4; e++) bv[e] = ld4(S + (x0 + 4 * k4 + e) * kLS + 32 + 4 * cg);
            fma24(z, av, bv);
        }
#pragma unroll
        for (int r = 0; r < 2; r++) st4(S + (t0 + rg + 8 * r) * kLS + s0 + 4 * cg, -z[r][0], -z[r][1], -z[r][2], -z[r][3]);
    }
    named_bar(bar_id, 64);   // T11 and T22 complete
    // the unit: lane (rg, cg) of the pair takes rows 8r + rg (r = 0..3) and
    // columns 4cg .. 4cg + 3 of a 32 x 32 block
    const int rg = (32 * role + l) >> 3, cg = l & 7;
    {
        float x[4][4] = {};   // X = A21 T11 into the upper-right block
#pragma unroll 2
        for (int k4 = 0; k4 < 8; k4++) {
            float4 av[4], bv[4];
#pragma unroll
            for (int r = 0; r < 4; r++) av[r] = ld4(S + (32 + 8 * r + rg) * kLS + 4 * k4);
#pragma unroll
            for (int e = 0; e < 4; e++) bv[e] = ld4(S + (4 * k4 + e) * kLS + 4 * cg);
            fma44(x, av, bv);
        }
#pragma unroll
        for (int r = 0; r < 4; r++) st4(S + (8 * r + rg) * kLS + 32 + 4 * cg, x[r][0], x[r][1], x[r][2], x[r][3]);
    }
    named_bar(bar_id, 64);   // X complete; A21 no longer read
    {
        float z[4][4] = {};   // T21 = -T22 X over A21
#pragma unroll 2
        for (int k4 = 0; k4 < 8; k4++) {
            float4 av[4], bv[4];
#pragma unroll
            for (int r = 0; r < 4; r++) av[r] = ld4(S + (32 + 8 * r + rg) * kLS + 32 + 4 * k4);
#pragma unroll
            for (int e = 0; e < 4; e++) bv[e] = ld4(S + (4 * k4 + e) * kLS + 32 + 4 * cg);
            fma44(z, av, bv);
        }
#pragma unroll
        for (int r = 0; r < 4; r++)
            st4(S + (32 + 8 * r + rg) * kLS + 4 * cg, -z[r][0], -z[r][1], -z[r][2], -z[r][3]);
    }
    named_bar(bar_id, 64);   // T complete in S
    store_tiles(S, dst, beta, gam, 8 * role, 8);
    if (tdst) store_t_f32(S, tdst, role);
}

}  // namespace tc
}  // namespace cpdr
