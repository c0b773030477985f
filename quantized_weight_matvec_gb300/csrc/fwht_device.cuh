// fwht_device.cuh -- device pieces of the Walsh-Hadamard transform shared by
// the CQ kernels (prepare, row gather) and the Hadamard MLP block.
//
// Method: needle.js tutorial "Inference engine, part 2: kernels and token
// step", section 1: the unnormalised in-place butterfly, strides 1, 2, 4, ...
// ascending, pair (i, i+h) -> (a+b, a-b), every result a float32; section 2:
// normalisation by 1/sqrt(n) computed in float64, the product taken in
// float64 and stored as float32.
#pragma once

#include <cuda_runtime.h>

namespace qmv {
namespace {

// RN32(RN64(v * s)): the page multiplies a float32 element by the float64
// 1/sqrt(group) and stores the product into float32.
__device__ __forceinline__ float scale_f64(float v, double s) {
    return __double2float_rn(__dmul_rn(double(v), s));
}

// Unnormalised FWHT of one group spread over a warp.  For G >= 32 each lane
// holds E = G/32 consecutive elements (element i = lane*E + e); for G < 32
// (E == 1) the warp holds 32/G groups, element i = lane % G.  Stride h is
// in-register while h < E, else a shuffle with lane distance h/E; the lane
// owning the lower index keeps a+b, the upper one keeps a-b.
template <int E>
__device__ __forceinline__ void fwht_warp(float (&v)[E], int G, int lane) {
    constexpr unsigned kAll = 0xffffffffu;
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int e = 0; e < E; e++) {
            if ((e & h) == 0) {
                float a = v[e], b = v[e + h];
                v[e] = __fadd_rn(a, b);
                v[e + h] = __fsub_rn(a, b);
            }
        }
    }
    for (int d = 1; d * E < G; d <<= 1) {
        bool upper = (lane & d) != 0;
#pragma unroll
        for (int e = 0; e < E; e++) {
            float o = __shfl_xor_sync(kAll, v[e], d);
            v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
        }
    }
}

}  // namespace
}  // namespace qmv
