// device_common.cuh -- small device helpers shared by the F8, I8 and
// int8-activation kernels.
#pragma once

#include <stdint.h>

namespace qmv {
namespace dev {

constexpr unsigned kFullMask = 0xffffffffu;

// E8M0 scale byte -> 2^(e-127) as float32 (ds4f-disk issue #6, step 1: the
// E8M0 block scales); e = 0 is the subnormal 2^-127, kept (no flush), and
// code 255 is NaN (the OCP microscaling convention).
__device__ __forceinline__ float e8m0(unsigned e) {
    if (e == 0) return __uint_as_float(0x00400000u);
    if (e == 255) return __uint_as_float(0x7fc00000u);
    return __uint_as_float(e << 23);
}

// Fixed-order butterfly sum over the warp; every lane ends with the same bits
// (a + b == b + a).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(kFullMask, v, d);
    return v;
}

// Streaming 16-byte load of read-only weights, not kept in L1.  Not volatile:
// the weights are never written while a matvec runs, so the compiler may
// schedule these loads freely.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 d;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
        : "l"(p));
    return d;
}

// cp.async: a 16-byte global -> shared copy that holds no registers (L2
// only), its commit, and a wait for all but the N most recent groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace dev
}  // namespace qmv
