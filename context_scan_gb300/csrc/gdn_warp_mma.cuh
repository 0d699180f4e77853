// gdn_warp_mma.cuh -- warp-level tensor-core tiles (mma.sync m16n8k8, tf32 operands, fp32
// accumulation) whose fragments are read straight from fp32 matrices in shared memory, for the
// backward kernels. Included by one translation unit per kernel family; internal linkage.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace {

// a tf32 operand rounded to nearest: the tensor core reads the top 19 bits, and adding half a
// tf32 unit to the sign-magnitude pattern carries into them
__device__ __forceinline__ uint32_t tf(float x) { return __float_as_uint(x) + 0x1000u; }

__device__ __forceinline__ void mma8(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc (a warp's MT x NT fragments of 16 x 8 at rows m0.., columns n0..) += A B over the
// contraction index 0 .. kd-1, with A(row, k) = fa(row, k) and B(k, col) = fb(k, col).
// Fragment layout (m16n8k8, tf32): lane = 4 g + t; A holds (g, t), (g+8, t), (g, t+4),
// (g+8, t+4); B holds (t, g), (t+4, g); the accumulator (g, 2t), (g, 2t+1), (g+8, 2t),
// (g+8, 2t+1).
template <int MT, int NT, class FA, class FB>
__device__ __forceinline__ void wtile(float (&acc)[MT][NT][4], int m0, int n0, int kd, int lane,
                                      FA fa, FB fb) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll 2
    for (int k0 = 0; k0 < kd; k0 += 8) {
        uint32_t a[MT][4], b[NT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int r = m0 + 16 * mt + g;
            a[mt][0] = tf(fa(r, k0 + t));
            a[mt][1] = tf(fa(r + 8, k0 + t));
            a[mt][2] = tf(fa(r, k0 + t + 4));
            a[mt][3] = tf(fa(r + 8, k0 + t + 4));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c = n0 + 8 * nt + g;
            b[nt][0] = tf(fb(k0 + t, c));
            b[nt][1] = tf(fb(k0 + t + 4, c));
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma8(acc[mt][nt], a[mt], b[nt]);
    }
}

// f(row, col, value&) for every accumulator element of the warp
template <int MT, int NT, class F>
__device__ __forceinline__ void wtile_each(float (&acc)[MT][NT][4], int m0, int n0, int lane, F f) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f(m0 + 16 * mt + g + 8 * (e >> 1), n0 + 8 * nt + 2 * t + (e & 1), acc[mt][nt][e]);
}

// sum over the four lanes that share g (the columns of one fragment row)
__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}
// sum over the eight lanes that share t (the rows of one fragment column)
__device__ __forceinline__ float col_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return x;
}

}  // namespace
}  // namespace gdn
