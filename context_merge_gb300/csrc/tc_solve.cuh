// One-warp solve of the per-chunk WY inverse, shared by the WY build of the
// scalar-gate path (tc_wy.cu) and the per-dim-gate preparation (tc_kda.cu).
#pragma once
#include <cuda_bf16.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"

namespace cpdr {
namespace tc {

constexpr int kLS = 68;   // row stride (floats) of the A scratch

// One warp: T = (I + A)^-1 of the 64 x 64 unit lower-triangular matrix whose
// strictly lower part A is in S[64][68] (zeros elsewhere), by rows:
//   T_ij = delta_ij - sum_{k < i} A_ik T_kj.
// Lane l keeps x1[i] = T_il (i = 0..63) and x2[m] = T_{32+m, 32+l} (m = 0..31;
// T_{i, 32+l} = 0 for i < 32).  Then writes T' = T diag(beta) and
// T'' = T diag(beta gamma) (hi, lo) as bf16 into the unit's three tiles.
__device__ __forceinline__ void solve_unit(const float *S, uint8_t *dst, const float *beta, const float *gam) {
    const int l = threadIdx.x & 31;
    float x1[64], x2[32];
#pragma unroll
    for (int i = 0; i < 64; i++) {
        float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k4 = 0; k4 < 16; k4++) {   // constant trip count: x1, x2 stay in registers
            if (4 * k4 >= i) break;
            const float4 a = *reinterpret_cast<const float4 *>(S + i * kLS + 4 * k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int k = 4 * k4 + e;
                if (k < i) {
                    a1[e] = fmaf(av[e], x1[k], a1[e]);
                    if (k >= 32) a2[e] = fmaf(av[e], x2[k - 32], a2[e]);
                }
            }
        }
        x1[i] = (i == l ? 1.f : 0.f) - ((a1[0] + a1[1]) + (a1[2] + a1[3]));
        if (i >= 32) x2[i - 32] = (i - 32 == l ? 1.f : 0.f) - ((a2[0] + a2[1]) + (a2[2] + a2[3]));
    }
    // column scales of this lane's two columns
    const float b1 = beta[l], b2 = beta[32 + l];
    const float c1 = b1 * gam[l], c2 = b2 * gam[32 + l];
    const uint32_t co1 = (uint32_t)(l & 7) * 2, q1 = (uint32_t)(l >> 3);
#pragma unroll
    for (int i = 0; i < 64; i++) {
        const float t1 = x1[i], t2 = i >= 32 ? x2[i - 32] : 0.f;
        const uint32_t o1 = sw128(i, q1) + co1, o2 = sw128(i, 4 + q1) + co1;
        const float u1 = t1 * b1, u2 = t2 * b2;
        const float w1 = t1 * c1, w2 = t2 * c2;
        const __nv_bfloat16 h1 = __float2bfloat16_rn(w1), h2 = __float2bfloat16_rn(w2);
        *reinterpret_cast<__nv_bfloat16 *>(dst + o1) = __float2bfloat16_rn(u1);
        *reinterpret_cast<__nv_bfloat16 *>(dst + o2) = __float2bfloat16_rn(u2);
        *reinterpret_cast<__nv_bfloat16 *>(dst + kWyTileBytes + o1) = h1;
        *reinterpret_cast<__nv_bfloat16 *>(dst + kWyTileBytes + o2) = h2;
        *reinterpret_cast<__nv_bfloat16 *>(dst + 2 * kWyTileBytes + o1) =
            __float2bfloat16_rn(w1 - __bfloat162float(h1));
        *reinterpret_cast<__nv_bfloat16 *>(dst + 2 * kWyTileBytes + o2) =
            __float2bfloat16_rn(w2 - __bfloat162float(h2));
    }
}

}  // namespace tc
}  // namespace cpdr
