// f8_common.cuh -- definitions shared by the F8 kernel files (f8_kernels.cu:
// batch 1 and the float kernels; f8_mma_kernels.cu: batch 2..8 on the tensor
// cores).
//
// Method: ds4f-disk issue #6 "attention + tokenizer + sampling" -- work item 1
// and step 1 (ds4f_f8_matvec: E4M3 decode with e=0 subnormal and the e=15
// clamp at 448; E8M0 block scales, scale [SR x SC] over weight [R x C], element
// (r, c) -> scale[r*SR/R][c*SC/C]).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "device_common.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace f8 {

constexpr unsigned kFull = 0xffffffffu;

// One partial argmax result: the best (value, row) a block found for a vector.
struct ArgBest {
    float v;
    int32_t pad;
    int64_t i;
};

struct F8Args {
    const uint8_t *w;
    const uint8_t *scale;
    const float *x;
    float *y;  // may be NULL for the argmax variant (then not stored)
    int64_t R, C, SR, SC;
    // argmax variant: [gridDim.x, B] partial results, the blocks' arrival
    // counter (zero between calls) and the final outputs
    ArgBest *ws;
    unsigned *ctr;
    int64_t *out_index;
    float *out_value;
};

// Total order of the greedy choice: NaN above every number (as numpy and
// torch argmax), larger values above smaller, then the lower row.
__device__ __forceinline__ bool arg_better(float av, int64_t ai, float bv, int64_t bi) {
    const bool an = isnan(av), bn = isnan(bv);
    if (an != bn) return an;
    if (!an && av != bv) return av > bv;
    return ai < bi;
}

// Per-warp running best for each vector (every lane holds the same values).
template <int B>
struct WarpBest {
    float v[B];
    int64_t i[B];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int k = 0; k < B; k++) {
            v[k] = -INFINITY;
            i[k] = INT64_MAX;
        }
    }
    __device__ __forceinline__ void offer(int k, float val, int64_t row) {
        if (arg_better(val, row, v[k], i[k])) {
            v[k] = val;
            i[k] = row;
        }
    }
};

// Block-level reduction of the warps' bests, written to ws[blockIdx.x * B + k].
// Every thread of the block must call it.
template <int B>
__device__ __forceinline__ void block_best_store(const WarpBest<B> &wb, ArgBest *ws) {
    __shared__ float sv[32][B];
    __shared__ int64_t si[32][B];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < B; k++) {
            sv[warp][k] = wb.v[k];
            si[warp][k] = wb.i[k];
        }
    }
    __syncthreads();
    if (threadIdx.x < B) {
        const int k = threadIdx.x;
        float bv = sv[0][k];
        int64_t bi = si[0][k];
        for (int w2 = 1; w2 < nw; w2++)
            if (arg_better(sv[w2][k], si[w2][k], bv, bi)) {
                bv = sv[w2][k];
                bi = si[w2][k];
            }
        ArgBest r;
        r.v = bv;
        r.pad = 0;
        r.i = bi;
        ws[int64_t(blockIdx.x) * B + k] = r;
    }
}

// Completion of the argmax, called by every thread of every block once the
// block's partial bests are stored in ws[blockIdx.x * B + k].  Each block
// makes its partials visible device-wide and counts itself in; the last
// block to arrive (the counter then wraps back to zero, ready for the next
// call) reduces all gridDim.x * B partials and writes the outputs.  The
// vectors go in rounds of vpr = min(B, warps) vectors, vector k0 + j of a
// round taking warps [j wpv, (j + 1) wpv) with wpv = warps / vpr; each
// thread loads its partials four at a time from L2 before comparing them,
// then shuffles and a shared-memory pass reduce them.  The order of
// arg_better is total, so the result is the greatest element whatever the
// order of reduction.
//
// `scratch` is shared memory of at least sizeof(ArgScratch) bytes, 8-byte
// aligned, that no thread touches after the kernel's last barrier before
// this call (the tensor-core kernels pass their epilogue buffer, so their
// dynamic shared-memory layout keeps its alignment).
struct ArgScratch {
    int64_t si[32];
    float sv[32];
    unsigned is_last;
};

__device__ __forceinline__ void argmax_complete(const F8Args &a, int B, void *scratch) {
    ArgScratch &sc = *static_cast<ArgScratch *>(scratch);
    int64_t *si = sc.si;
    float *sv = sc.sv;
    // the barrier orders the block's partial stores before thread 0's fence,
    // which makes them visible device-wide before the count (and, in the
    // last block, orders the count before the reads of every partial)
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        sc.is_last = (atomicInc(a.ctr, gridDim.x - 1) == gridDim.x - 1) ? 1u : 0u;
        __threadfence();
    }
    __syncthreads();
    if (!sc.is_last) return;  // block-uniform
    const int nblocks = int(gridDim.x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = int(blockDim.x >> 5);
    const int vpr = B < nw ? B : nw;
    const int wpv = nw / vpr;
    const int j = warp / wpv, sub = warp - j * wpv;
    const int stride = wpv * 32, first = sub * 32 + lane;
    for (int k0 = 0; k0 < B; k0 += vpr) {
        const int k = k0 + j;
        float bv = -INFINITY;
        int64_t bi = INT64_MAX;
        if (j < vpr && k < B) {  // warp-uniform
            for (int b0 = first; b0 < nblocks; b0 += 4 * stride) {
                ArgBest e[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int b = b0 + q * stride;
                    if (b < nblocks) {
                        const ArgBest *src = a.ws + int64_t(b) * B + k;
                        e[q].v = __ldcg(&src->v);
                        e[q].i = __ldcg(&src->i);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int b = b0 + q * stride;
                    if (b < nblocks && arg_better(e[q].v, e[q].i, bv, bi)) {
                        bv = e[q].v;
                        bi = e[q].i;
                    }
                }
            }
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, d);
            const int64_t oi = __shfl_xor_sync(kFull, bi, d);
            if (arg_better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            sv[warp] = bv;
            si[warp] = bi;
        }
        __syncthreads();
        if (int(threadIdx.x) < vpr && k0 + int(threadIdx.x) < B) {
            const int jj = threadIdx.x;
            float v = sv[jj * wpv];
            int64_t i = si[jj * wpv];
            for (int w2 = 1; w2 < wpv; w2++)
                if (arg_better(sv[jj * wpv + w2], si[jj * wpv + w2], v, i)) {
                    v = sv[jj * wpv + w2];
                    i = si[jj * wpv + w2];
                }
            a.out_index[k0 + jj] = i;
            a.out_value[k0 + jj] = v;
        }
        __syncthreads();
    }
}

// E4M3 byte -> float32 from its fields, with the saturation at 448 (so the
// codes 0x7F / 0xFF, NaN in the OCP "fn" variant, read as +/-448).
__device__ __forceinline__ float e4m3_exact(unsigned b) {
    const unsigned e = (b >> 3) & 15u, m = b & 7u;
    float mag;
    if (e == 0) {
        mag = float(m) * 0.001953125f;  // m * 2^-9, exact
    } else {
        mag = __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) * 2^(e-7)
        mag = fminf(mag, 448.0f);
    }
    return (b & 0x80u) ? -mag : mag;
}

using dev::warp_sum;

// Exact per-element evaluation of one output, shared by the general kernel
// and by the fast kernel's fix-up of rows that hit a saturated code.  The
// whole warp calls it.
static __device__ float f8_row_exact(const F8Args &a, int64_t r, int v, const float *lut) {
    const int64_t rb = r * a.SR / a.R;
    const uint8_t *wr = a.w + r * a.C;
    const uint8_t *sr = a.scale + rb * a.SC;
    const float *xv = a.x + int64_t(v) * a.C;
    float acc = 0.0f;
    for (int64_t c = threadIdx.x & 31; c < a.C; c += 32) {
        const float wv = lut ? lut[__ldg(wr + c)] : e4m3_exact(__ldg(wr + c));
        const float sv = dev::e8m0(__ldg(sr + c * a.SC / a.C));
        acc = fmaf(wv * sv, __ldg(xv + c), acc);
    }
    return warp_sum(acc);
}

using dev::ld_stream;

__device__ __forceinline__ unsigned word_of(const uint4 &d, int q) {
    return q == 0 ? d.x : q == 1 ? d.y : q == 2 ? d.z : d.w;
}

// True when every `width`-column chunk maps to a single scale block: the
// first column of each block b, ceil(b*C/SC), is a multiple of `width`.
inline bool chunks_uniform(int64_t C, int64_t SC, int64_t width = 16) {
    for (int64_t b = 1; b < SC; b++) {
        const int64_t start = (b * C + SC - 1) / SC;
        if (start % width != 0) return false;
    }
    return true;
}


// The mma.sync tensor-core kernels (f8_mma_kernels.cu), for the batch 2..8
// calls the fifth-generation kernel does not take.  mma_fits: whether they take
// this call (batch >= 2, C % 64 == 0, C >= 256, 16-byte aligned w and x,
// 64-column-aligned scale blocks, shared memory in reach); launch_mma runs
// them (with the argmax epilogue when `am`), setting the grid size used.
bool mma_fits(const F8Args &a, int batch);
qmv_status launch_mma(const F8Args &a, int batch, bool am, cudaStream_t s, int &blocks_out);

// The fifth-generation tensor-core kernel (f8_tc_kernels.cu).  tc_fits:
// whether it takes this call (batch 5..8, C % 128 == 0 with C <= 4096, at
// least 3 64-row units per SM, 16-byte aligned w and x, every scale block
// starting on a multiple of 64 rows and of 128 columns, y given); launch_tc
// runs it.  tc_wait_timeouts
// reads how many of its waits have ever run out of time (none, normally).
bool tc_fits(const F8Args &a, int batch);
qmv_status launch_tc(const F8Args &a, int batch, bool am, cudaStream_t s, int &blocks_out);
qmv_status tc_wait_timeouts(unsigned long long *count);

}  // namespace f8
}  // namespace qmv
