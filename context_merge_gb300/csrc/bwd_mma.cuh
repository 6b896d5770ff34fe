// Warp-level tf32 tensor-core products from shared or global memory for the
// backward's input-gradient kernels: mma.sync m16n8k8 (fp32 accumulation)
// on operand views that give element (r, c) of a matrix.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace cpdr {
namespace bwdmm {

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// D += A * B on a 16 x 8 tile, tf32 operands (the fp32 bit pattern's top 19
// bits), fp32 accumulation
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Operand views: element (r, c) of a matrix in shared memory, fp32 or bf16,
// with row and column strides (a transposed view swaps them) and an
// optional per-row (or per-column) scale.
struct Fv {
    const float *p;
    int rs, cs;
    __device__ __forceinline__ float at(int r, int c) const { return p[r * rs + c * cs]; }
};
struct Bv {
    const __nv_bfloat16 *p;
    int rs, cs;
    __device__ __forceinline__ float at(int r, int c) const { return bf(p + r * rs + c * cs); }
};

// Warp tile: C (16 x 8 NTL) += A (rows m0.., K columns) * B (K rows, columns n0 + 8 nt ..).
template <int NTL, int K, typename AV, typename BV>
__device__ __forceinline__ void warp_mm(float (&c)[NTL][4], const AV &a, int m0, const BV &b, const int (&n0)[NTL]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t af[4];
        af[0] = __float_as_uint(a.at(m0 + g, k0 + t));
        af[1] = __float_as_uint(a.at(m0 + g + 8, k0 + t));
        af[2] = __float_as_uint(a.at(m0 + g, k0 + t + 4));
        af[3] = __float_as_uint(a.at(m0 + g + 8, k0 + t + 4));
#pragma unroll
        for (int nt = 0; nt < NTL; nt++) {
            uint32_t bfr[2];
            bfr[0] = __float_as_uint(b.at(k0 + t, n0[nt] + g));
            bfr[1] = __float_as_uint(b.at(k0 + t + 4, n0[nt] + g));
            mma_tf32(c[nt], af, bfr);
        }
    }
}

template <int N>
__device__ __forceinline__ void zero(float (&c)[N][4]) {
#pragma unroll
    for (int i = 0; i < N; i++) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
}

}  // namespace bwdmm
}  // namespace cpdr
