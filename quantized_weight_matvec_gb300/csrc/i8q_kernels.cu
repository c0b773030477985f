// i8q_kernels.cu -- int8 weights times int8 activations quantized per group
// of 32, sm_103a.
//
// Method: Mnemonic "In the browser", "Dot products and math": activations
// are quantized to int8 per group of 32 with one float scale per group, once
// per vector; the int8 x int8 dot products are exact int32 sums, which only
// then become floats scaled by the activation group's scale.  The weights
// are the I8 format of ds4f-disk issue #6, step 4 (int8 with one E8M0 scale
// per 16 consecutive columns of a row, [R, ceil(C/16)]).
//
//   quantize:  d[v][j] = m / 127 (m = max |x| over columns [32 j, 32 j + 32))
//              q[v][c] = clamp(rint(x[v][c] / d[v][c/32]), -127, 127)
//   matvec:    y[v][r] = sum_c w[r][c] * e8m0(scale[r][c/16]) * q[v][c] * d[v][c/32]
//
// Both divisions are IEEE float32 (__fdiv_rn) and rint rounds to nearest
// even, so the codes are exactly those of any IEEE float32 evaluation of the
// same definition.  d = 0 gives q = 0; a group holding Inf or NaN gives
// d = NaN and q = 0, so every output that group meets is NaN.
//
// The page's WebAssembly stores the codes widened to int16 because its SIMD
// has only an int16 dot product; dp4a multiplies int8 by int8 directly, so
// the codes stay int8 here.
//
// Matvec layout: a lane's 16-byte weight chunk (columns 16 ch .. 16 ch + 15)
// is one weight scale group and half of activation group ch / 2.  Per chunk
// and vector, four dp4a give the exact int32 sum S (|S| <= 16 * 128 * 127),
// which converts to float exactly; float(S) * e8m0 is exact too (a power of
// two, barring underflow), and one FMA adds it times d to the accumulator.
#include <stdint.h>

#include "device_common.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

struct I8QArgs {
    const int8_t *w;
    const uint8_t *scale;
    const int8_t *xq;
    const float *xd;
    float *y;
    int64_t R, C, SG, XG;  // SG = ceil(C/16) weight groups, XG = ceil(C/32) activation groups
};

using dev::warp_sum;

// ---------------------------------------------------------------------------
// Quantizer: one warp per (vector, group of 32); lane l holds column 32 j + l.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) i8_quantize_kernel(const float *x, int64_t C, int64_t ngroups,
                                                          int64_t jobs, int8_t *xq, float *xd) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (job >= jobs) return;  // warp-uniform
    const int64_t v = job / ngroups, g = job - v * ngroups;
    const int64_t c = g * 32 + lane;
    const bool in = c < C;
    const float xv = in ? __ldg(x + v * C + c) : 0.0f;
    const bool finite = __all_sync(kFull, isfinite(xv));
    float m = fabsf(xv);
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, s));
    const float d = finite ? __fdiv_rn(m, 127.0f) : __uint_as_float(0x7fc00000u);
    int code = 0;
    if (finite && d != 0.0f) {
        float t = rintf(__fdiv_rn(xv, d));
        t = fminf(fmaxf(t, -127.0f), 127.0f);
        code = int(t);
    }
    if (in) xq[v * C + c] = int8_t(code);
    if (lane == 0) xd[v * ngroups + g] = d;
}

// ---------------------------------------------------------------------------
// Streaming matvec (C % 16 == 0, 16-byte aligned w and xq).  Warps walk tiles
// of T rows in grid-stride order; per step a lane loads the 16-byte chunk
// ch = base + lane + 32 st of each of the T rows, NSTEP steps at a time
// (NSTEP = 1 for large matrices, more when too few tiles keep the grid busy).
// The codes and scales of all vectors are staged in shared memory once per
// block: xs[v][C] int8 (lane reads of 16 consecutive bytes: conflict-free),
// ds[v][XG] float (lanes 2k, 2k+1 share a word: broadcast).
// ---------------------------------------------------------------------------
template <int T>
__device__ __forceinline__ void load_rows(uint4 (&d)[T], unsigned (&e)[T], const I8QArgs &a, int64_t r0,
                                          int rows, int64_t ch, int64_t nchunk) {
    const int64_t chc = ch < nchunk ? ch : nchunk - 1;
#pragma unroll
    for (int t = 0; t < T; t++) {
        const int64_t r = r0 + (t < rows ? t : rows - 1);
        asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
            : "=r"(d[t].x), "=r"(d[t].y), "=r"(d[t].z), "=r"(d[t].w)
            : "l"(a.w + r * a.C + chc * 16));
        e[t] = __ldg(a.scale + r * a.SG + chc);
    }
}

template <int B, int T, int NSTEP>
__global__ void __launch_bounds__(256) i8q_kernel(I8QArgs a) {
    extern __shared__ uint4 dsm[];
    int8_t *xs = reinterpret_cast<int8_t *>(dsm);
    float *ds = reinterpret_cast<float *>(xs + int64_t(B) * a.C);
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nchunk = a.C >> 4;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t ntiles = (a.R + T - 1) / T;
    int64_t tile = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;

    // the first weights in flight before the dependency wait (they never
    // depend on the preceding kernel) and while the codes are staged
    uint4 w[NSTEP][T];
    unsigned e[NSTEP][T];
    if (tile < ntiles) {
        const int rows = int(min(int64_t(T), a.R - tile * T));
#pragma unroll
        for (int st = 0; st < NSTEP; st++) load_rows<T>(w[st], e[st], a, tile * T, rows, lane + 32 * st, nchunk);
    }
    pdl_wait();
    {
        const int64_t nv = (int64_t(B) * a.C) >> 4;
        const uint4 *src = reinterpret_cast<const uint4 *>(a.xq);
        for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) dsm[i] = __ldg(src + i);
        const int64_t nd = int64_t(B) * a.XG;
        for (int64_t i = threadIdx.x; i < nd; i += blockDim.x) ds[i] = __ldg(a.xd + i);
    }
    __syncthreads();

    float acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) acc[t][v] = 0.0f;
    for (; tile < ntiles; tile += nwarps) {
        const int64_t r0 = tile * T;
        const int rows = int(min(int64_t(T), a.R - r0));
        for (int64_t base = 0; base < nchunk; base += 32 * NSTEP) {
            if (base != 0) {
#pragma unroll
                for (int st = 0; st < NSTEP; st++) load_rows<T>(w[st], e[st], a, r0, rows, base + lane + 32 * st, nchunk);
            }
#pragma unroll
            for (int st = 0; st < NSTEP; st++) {
                const int64_t ch = base + lane + 32 * st;
                if (ch >= nchunk) continue;
                float sw[T];
#pragma unroll
                for (int t = 0; t < T; t++) sw[t] = dev::e8m0(e[st][t]);
#pragma unroll
                for (int v = 0; v < B; v++) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xs + int64_t(v) * a.C + ch * 16);
                    const float dv = ds[int64_t(v) * a.XG + (ch >> 1)];
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        int s = __dp4a(int(w[st][t].x), int(xv.x), 0);
                        s = __dp4a(int(w[st][t].y), int(xv.y), s);
                        s = __dp4a(int(w[st][t].z), int(xv.z), s);
                        s = __dp4a(int(w[st][t].w), int(xv.w), s);
                        acc[t][v] = fmaf(__int2float_rn(s) * sw[t], dv, acc[t][v]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < T; t++)
#pragma unroll
            for (int v = 0; v < B; v++) {
                const float val = warp_sum(acc[t][v]);
                acc[t][v] = 0.0f;
                if (t < rows && lane == 0) a.y[int64_t(v) * a.R + r0 + t] = val;
            }
        // next tile's first steps
        const int64_t nt = tile + nwarps;
        if (nt < ntiles) {
            const int nrows = int(min(int64_t(T), a.R - nt * T));
#pragma unroll
            for (int st = 0; st < NSTEP; st++) load_rows<T>(w[st], e[st], a, nt * T, nrows, lane + 32 * st, nchunk);
        }
    }
}

// ---------------------------------------------------------------------------
// General kernel: any C and alignment.  One warp per row, one column per
// lane step: the exact integer product w * q times the two scales.
// ---------------------------------------------------------------------------
template <int B>
__global__ void __launch_bounds__(256) i8q_general_kernel(I8QArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < a.R; r += nwarps) {
        const int8_t *wr = a.w + r * a.C;
        const uint8_t *sr = a.scale + r * a.SG;
        float acc[B];
#pragma unroll
        for (int v = 0; v < B; v++) acc[v] = 0.0f;
        for (int64_t c = lane; c < a.C; c += 32) {
            const int wv = __ldg(wr + c);
            const float s = dev::e8m0(__ldg(sr + (c >> 4)));
#pragma unroll
            for (int v = 0; v < B; v++) {
                const int p = wv * int(__ldg(a.xq + int64_t(v) * a.C + c));
                acc[v] = fmaf(float(p) * s, __ldg(a.xd + int64_t(v) * a.XG + (c >> 5)), acc[v]);
            }
        }
#pragma unroll
        for (int v = 0; v < B; v++) {
            const float val = warp_sum(acc[v]);
            if (lane == 0) a.y[int64_t(v) * a.R + r] = val;
        }
    }
}

// Shared memory of i8q_kernel: the codes and scales of all B vectors.
inline size_t stage_bytes(int B, int64_t C) {
    const int64_t xg = (C + 31) / 32;
    return size_t(B) * size_t(C) + size_t(B) * size_t(xg) * 4;
}
constexpr size_t kStageMax = 160 * 1024;

template <int B, int T, int NSTEP>
qmv_status launch_stream(const I8QArgs &a, cudaStream_t s) {
    const size_t smem = stage_bytes(B, a.C);
    auto kern = i8q_kernel<B, T, NSTEP>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int blocks = grid_blocks(kp, 256, smem, (a.R + T - 1) / T);
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(256), smem, s, a));
}

template <int B>
qmv_status launch_i8q(const I8QArgs &a, cudaStream_t s) {
    const bool fast = (a.C % 16 == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(a.xq) % 16 == 0) && stage_bytes(B, a.C) <= kStageMax;
    if (!fast) {
        const void *kp = reinterpret_cast<const void *>(i8q_general_kernel<B>);
        const int blocks = grid_blocks(kp, 256, 0, a.R);
        return from_cuda(launch_pdl(i8q_general_kernel<B>, dim3(unsigned(blocks)), dim3(256), 0, s, a));
    }
    constexpr int T = (B <= 2) ? 8 : (B <= 4 ? 4 : 2);
    const void *kp = reinterpret_cast<const void *>(i8q_kernel<B, T, 1>);
    const int64_t capacity = int64_t(occupancy(kp, 256, stage_bytes(B, a.C))) * sm_count() * 8;
    // too few tiles for a streaming grid: shorter tiles, several steps per load
    if ((a.R + T - 1) / T < 4 * capacity) return launch_stream<B, 2, (B <= 2) ? 8 : 4>(a, s);
    // A streaming matrix from batch 4 on: the dp4a and float work per weight
    // outgrows the weight stream, so the I8 tensor-core kernel takes the call
    // when it fits, with the activations q * d split into f16 hi + lo like
    // float x.
    if (B >= 4) {
        qmv_status st = QMV_OK;
        if (launch_i8_matvec_q8_mma(a.w, a.R, a.C, a.scale, a.xq, a.xd, B, a.y, s, st)) return st;
    }
    return launch_stream<B, T, 1>(a, s);
}

}  // namespace

qmv_status launch_i8_quantize_x(const float *x, int64_t C, int batch, int8_t *xq, float *xd, cudaStream_t s) {
    const int64_t ngroups = (C + 31) / 32, jobs = int64_t(batch) * ngroups;
    const int64_t blocks = (jobs + 7) / 8;
    return from_cuda(launch_pdl(i8_quantize_kernel, dim3(unsigned(blocks)), dim3(256), 0, s, x, C, ngroups, jobs,
                                xq, xd));
}

qmv_status launch_i8_matvec_q8(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale, const int8_t *xq,
                               const float *xd, int batch, float *y, cudaStream_t s) {
    I8QArgs a{w, scale, xq, xd, y, R, C, (C + 15) / 16, (C + 31) / 32};
    switch (batch) {
        case 1: return launch_i8q<1>(a, s);
        case 2: return launch_i8q<2>(a, s);
        case 3: return launch_i8q<3>(a, s);
        case 4: return launch_i8q<4>(a, s);
        case 5: return launch_i8q<5>(a, s);
        case 6: return launch_i8q<6>(a, s);
        case 7: return launch_i8q<7>(a, s);
        default: return launch_i8q<8>(a, s);
    }
}

}  // namespace qmv
