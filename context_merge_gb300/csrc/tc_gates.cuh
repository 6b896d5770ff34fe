// In-chunk gate scan shared by the WY build and the chain kernels, so that
// both derive bit-identical cumulative gates from the same inputs.
//
// Gates are natural-log g = log(alpha) (fp32); the kernels work in log2 units
// with exp2, as the article's kernels do with chunk_local_cumsum(..., scale =
// RCP_LN2) ([FLA-CP] §4).
#pragma once

#include <cuda_runtime.h>

namespace cpdr {
namespace tc {

constexpr float kLog2e = 1.4426950408889634f;
// Factored in-chunk exponentials 2^(G_i - G_j) = e_i f_j (e, f taken around
// row 31) are used while every |G_i - G_31| stays within this bound; beyond
// it the kernels evaluate 2^(G_i - G_j) directly.
constexpr float kFactorBound = 100.f;

// One warp scans one 64-row chunk: lane l holds rows 2l and 2l+1 with log2
// gates g0, g1 (padded rows carry 0).
struct LaneGates {
    float G0, G1;   // inclusive cumulative log2 gates of rows 2l, 2l+1
    float GC;       // the chunk total G_63
    float Gr;       // reference G_31 of the factored exponentials
    bool exact;     // the span around Gr exceeds kFactorBound
};

__device__ __forceinline__ LaneGates scan_gates(float g0, float g1) {
    const int lane = threadIdx.x & 31;
    float x = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    LaneGates r;
    r.G1 = x;
    r.G0 = x - g1;
    r.GC = __shfl_sync(0xffffffffu, x, 31);
    r.Gr = __shfl_sync(0xffffffffu, r.G1, 15);
    float span = fmaxf(fabsf(r.G0 - r.Gr), fabsf(r.G1 - r.Gr));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) span = fmaxf(span, __shfl_xor_sync(0xffffffffu, span, o));
    r.exact = span > kFactorBound;
    return r;
}

}  // namespace tc
}  // namespace cpdr
