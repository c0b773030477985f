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
#include <math.h>

namespace qmv {
namespace {

// RN32(RN64(v * s)): the page multiplies a float32 element by the float64
// 1/sqrt(group) and stores the product into float32.
__device__ __forceinline__ float scale_f64(float v, double s) {
    return __double2float_rn(__dmul_rn(double(v), s));
}

// The same value without float64 arithmetic (GB300 issues about two
// float64 multiplies per clock per SM).  s = s1 + s2 + s3 exactly, each a
// float32; then p = RN32(v s1), its exact error e = v s1 - p (one FMA),
// t = RN32(RN32(v s2 + e) + v s3) by two FMAs, and the result RN32(p + t).
// For s = RN64(1/sqrt 2) * 2^-k (group or dimension an odd power of two)
// this equals RN32(RN64(v * s)) for every float32 mantissa, both signs
// (checked exhaustively on the host against the definition), as long as no
// step leaves the normal range; for s = 2^-k it is v * s exactly.  Other s,
// and nonzero |v| outside [2^-60, 2^100] (tiny, huge, Inf, NaN), take the
// float64 product.
struct Scale {
    double s;           // RN64(1/sqrt(n))
    float s1, s2, s3;   // s = s1 + s2 + s3
    int fast;           // s is 2^-k or RN64(1/sqrt 2) * 2^-k
};

inline Scale make_scale(double s) {
    Scale k;
    k.s = s;
    k.s1 = float(s);
    const double r = s - double(k.s1);
    k.s2 = float(r);
    k.s3 = float(r - double(k.s2));
    int e1 = 0, e2 = 0;
    const double m1 = frexp(s, &e1);                     // s = m1 * 2^e1, m1 in [0.5, 1)
    const double m2 = frexp(s / (1.0 / sqrt(2.0)), &e2);  // exact when s = that constant * 2^-k
    const bool exact_split = double(k.s1) + double(k.s2) + double(k.s3) == s;
    k.fast = exact_split && s > 0.0 && (m1 == 0.5 || (m2 == 0.5 && s == ldexp(1.0 / sqrt(2.0), e2 - 1)))
                 ? 1
                 : 0;
    return k;
}

// (out of line, so that the compiler does not predicate the float64
// multiply into the common path)
__device__ __noinline__ float scale_f64_rare(float v, double s) { return scale_f64(v, s); }

// Whether v takes the float32 form: zero, or |v| in [2^-60, 2^100].
__device__ __forceinline__ bool scale_in_range(float v) {
    const float av = fabsf(v);
    return av == 0.0f || (av >= 0x1p-60f && av <= 0x1p100f);
}

// The float32 form.  copysign keeps the sign of a zero product (p + t would
// give +0 for v = -0); for every other v in range |t| < |p| / 2, so it
// changes nothing.
__device__ __forceinline__ float scale_f32(float v, const Scale &k) {
    const float p = __fmul_rn(v, k.s1);
    const float e = __fmaf_rn(v, k.s1, -p);
    float t = __fmaf_rn(v, k.s2, e);
    t = __fmaf_rn(v, k.s3, t);
    return copysignf(__fadd_rn(p, t), p);
}

__device__ __forceinline__ float scale_rn(float v, const Scale &k) {
    if (__builtin_expect(k.fast && scale_in_range(v), 1)) return scale_f32(v, k);
    return scale_f64_rare(v, k.s);
}

// scale_rn of E values with one test for all of them (one branch per
// group of values, not one per value).
template <int E>
__device__ __forceinline__ void scale_rn_all(float (&v)[E], const Scale &k) {
    bool ok = k.fast != 0;
#pragma unroll
    for (int e = 0; e < E; e++) ok = ok && scale_in_range(v[e]);
    if (__builtin_expect(ok, 1)) {
#pragma unroll
        for (int e = 0; e < E; e++) v[e] = scale_f32(v[e], k);
    } else {
#pragma unroll
        for (int e = 0; e < E; e++) v[e] = scale_rn(v[e], k);
    }
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
