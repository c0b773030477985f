// f8_kernels.cu -- block-scaled F8 E4M3 matvec for sm_103a.
//
// Method: ds4f-disk issue #6 "attention + tokenizer + sampling" -- work item 1
// and step 1 (ds4f_f8_matvec: E4M3 decode with e=0 subnormal and the e=15
// clamp at 448; E8M0 block scales, scale [SR x SC] over weight [R x C], element
// (r, c) -> scale[r*SR/R][c*SC/C]), work item 3 (the ~246k x 4096 head, the
// largest matvec, kept resident).  The page's kernels are scalar / NEON / AVX2
// loops with a byte lookup table; here the weight stream is the whole cost,
// so the fast kernel is built around 128-bit streaming loads and keeps every
// other operand on chip.
//
//   y[v][r] = sum_c E4M3(w[r][c]) * E8M0(scale[r*SR/R][c*SC/C]) * x[v][c]
//
// E8M0 code 255 is read as NaN (OCP microscaling); every other code is
// 2^(e-127), exact in float32 (e = 0 is the subnormal 2^-127).
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "qmv_internal.h"

namespace qmv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

struct F8Args {
    const uint8_t *w;
    const uint8_t *scale;
    const float *x;
    float *y;
    int64_t R, C, SR, SC;
};

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

// E8M0 byte -> 2^(e-127) as float32; 255 -> NaN.
__device__ __forceinline__ float e8m0_value(unsigned e) {
    if (e == 0) return __uint_as_float(0x00400000u);  // 2^-127, subnormal
    if (e == 255) return __uint_as_float(0x7fc00000u);
    return __uint_as_float(e << 23);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;  // every lane holds the same bits (a + b == b + a)
}

// Exact per-element evaluation of one output, shared by the general kernel
// and by the fast kernel's fix-up of rows that hit a saturated code.  The
// whole warp calls it.
__device__ float f8_row_exact(const F8Args &a, int64_t r, int v, const float *lut) {
    const int64_t rb = r * a.SR / a.R;
    const uint8_t *wr = a.w + r * a.C;
    const uint8_t *sr = a.scale + rb * a.SC;
    const float *xv = a.x + int64_t(v) * a.C;
    float acc = 0.0f;
    for (int64_t c = threadIdx.x & 31; c < a.C; c += 32) {
        const float wv = lut ? lut[__ldg(wr + c)] : e4m3_exact(__ldg(wr + c));
        const float sv = e8m0_value(__ldg(sr + c * a.SC / a.C));
        acc = fmaf(wv * sv, __ldg(xv + c), acc);
    }
    return warp_sum(acc);
}

// ---------------------------------------------------------------------------
// General kernel: any C, any scale blocking, any alignment.  One warp per
// row, a shared-memory table of the 256 exact E4M3 values.
// ---------------------------------------------------------------------------
template <int B>
__global__ void __launch_bounds__(256) f8_general_kernel(F8Args a) {
    __shared__ float lut[256];
    lut[threadIdx.x] = e4m3_exact(threadIdx.x);
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < a.R; r += nwarps) {
#pragma unroll 1
        for (int v = 0; v < B; v++) {
            const float val = f8_row_exact(a, r, v, lut);
            if (lane == 0) a.y[int64_t(v) * a.R + r] = val;
        }
    }
}

// ---------------------------------------------------------------------------
// Fast kernel.  Requirements (checked by the launcher): C % 16 == 0, w and x
// 16-byte aligned, and every 16-column chunk inside one scale block.
//
// Each warp owns an even share of the rows and walks it in tiles of T rows.
// Lane l takes the 16-byte chunks l, l+32, ... of every row in the tile, so
// one warp-wide load streams 512 contiguous bytes of a row and the T loads of
// a chunk are independent.  The (tile, chunk) loop is flattened and, with PF,
// the T loads of the next step (the next chunk, or the first chunk of the
// next tile) are issued before the current step is decoded, so every warp
// keeps 2 * T * 512 bytes of the weight stream in flight.
//
// For a tile whose rows share one scale row, x is multiplied by the chunk's
// E8M0 scale once and reused by all T rows; a tile straddling two scale rows
// scales x per row.  Decode: cvt.rn.f16x2.e4m3x2 (exact) then f16 -> f32
// (exact), one FMA per weight and vector, float32 accumulation and a
// fixed-order warp reduction.  The hardware conversion maps 0x7F / 0xFF to
// NaN; a row whose sum comes out NaN is recomputed exactly (saturating
// decode), which also keeps NaN scales and non-finite x consistent with the
// per-element definition.
// ---------------------------------------------------------------------------

// Streaming 16-byte load of read-only weights, not kept in L1.  Not volatile:
// the weights are never written while a matvec runs, so the compiler may
// schedule these loads freely.
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    uint4 d;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
        : "l"(p));
    return d;
}

__device__ __forceinline__ void decode4(unsigned word, float (&f)[4]) {
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(word & 0xffffu), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(word >> 16), __NV_E4M3);
    float2 a = __half22float2(__half2(lo));
    float2 b = __half22float2(__half2(hi));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
}

__device__ __forceinline__ unsigned word_of(const uint4 &d, int q) {
    return q == 0 ? d.x : q == 1 ? d.y : q == 2 ? d.z : d.w;
}

// The T weight chunks of one step: rows r0 .. r0+rows-1, chunk ch.  Rows past
// the tile's end re-read its last row and chunks past the row's end re-read
// its last chunk (in bounds, results unused), so no load is predicated.
template <int T>
__device__ __forceinline__ void load_step(uint4 (&d)[T], const F8Args &a, int64_t r0, int rows,
                                          int64_t ch, int64_t nchunk) {
    const int64_t chc = ch < nchunk ? ch : nchunk - 1;
    const uint8_t *p = a.w + r0 * a.C + chc * 16;
#pragma unroll
    for (int t = 0; t < T; t++) d[t] = ld_stream(p + int64_t(t < rows ? t : rows - 1) * a.C);
}

// acc[t][v] += sum over the 16 columns of chunk ch of w[t] * s * x[v].
// UNIFORM: every row of the tile uses the scale row srow0; otherwise row t
// uses srow0 + ((dpack >> 4t) & 15) * SC.
template <int B, int T, bool UNIFORM>
__device__ __forceinline__ void compute_step(float (&acc)[T][B], const uint4 (&d)[T], const F8Args &a,
                                             const uint8_t *srow0, uint32_t dpack, int cb, int64_t ch) {
    float s0 = 0.0f;
    if (UNIFORM) s0 = e8m0_value(__ldg(srow0 + cb));
#pragma unroll
    for (int q = 0; q < 4; q++) {
        float xv[B][4];
#pragma unroll
        for (int v = 0; v < B; v++) {
            const float4 x4 = __ldg(reinterpret_cast<const float4 *>(a.x + v * a.C + ch * 16 + 4 * q));
            xv[v][0] = x4.x;
            xv[v][1] = x4.y;
            xv[v][2] = x4.z;
            xv[v][3] = x4.w;
        }
        float xs[B][4];
        if (UNIFORM) {
#pragma unroll
            for (int v = 0; v < B; v++)
#pragma unroll
                for (int k = 0; k < 4; k++) xs[v][k] = xv[v][k] * s0;
        }
#pragma unroll
        for (int t = 0; t < T; t++) {
            if (!UNIFORM) {
                const float st = e8m0_value(__ldg(srow0 + int64_t((dpack >> (4 * t)) & 15u) * a.SC + cb));
#pragma unroll
                for (int v = 0; v < B; v++)
#pragma unroll
                    for (int k = 0; k < 4; k++) xs[v][k] = xv[v][k] * st;
            }
            float f[4];
            decode4(word_of(d[t], q), f);
#pragma unroll
            for (int v = 0; v < B; v++) {
                acc[t][v] = fmaf(f[0], xs[v][0], acc[t][v]);
                acc[t][v] = fmaf(f[1], xs[v][1], acc[t][v]);
                acc[t][v] = fmaf(f[2], xs[v][2], acc[t][v]);
                acc[t][v] = fmaf(f[3], xs[v][3], acc[t][v]);
            }
        }
    }
}

template <int B, int T, bool PF, bool GS>
__global__ void __launch_bounds__(256) f8_fast_kernel(F8Args a) {
    extern __shared__ int chunk_cb[];
    const int64_t nchunk = a.C >> 4;
    // (depends only on the shapes: runs before the wait)
    for (int64_t ch = threadIdx.x; ch < nchunk; ch += blockDim.x)
        chunk_cb[ch] = int((ch * 16 * a.SC) / a.C);
    pdl_wait();
    pdl_trigger();
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    // GS: tiles in grid-stride order (all warps sweep one region of the
    // matrix together); otherwise each warp owns an even contiguous share.
    const int64_t row_end = GS ? a.R : a.R * (wid + 1) / nwarps;
    int64_t r0 = GS ? wid * T : a.R * wid / nwarps;
    const int64_t tile_stride = GS ? nwarps * T : T;
    if (r0 >= row_end) return;
    const int iters = int((nchunk + 31) >> 5);

    int rows = int(min(int64_t(T), row_end - r0));
    int j = 0;
    uint4 cur[T];
    load_step<T>(cur, a, r0, rows, lane, nchunk);

    float acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) acc[t][v] = 0.0f;

    static_assert(T <= 8, "per-row scale deltas are packed in 4 bits");
    const uint8_t *srow0 = a.scale;
    uint32_t dpack = 0;
    bool uniform = true;
    auto setup_tile = [&]() {
        // rows of one tile span at most T + 1 scale rows (SR <= R), so each
        // row's offset from the first fits in 4 bits
        const int64_t rb0 = r0 * a.SR / a.R, rb1 = (r0 + rows - 1) * a.SR / a.R;
        uniform = (rb0 == rb1);
        srow0 = a.scale + rb0 * a.SC;
        dpack = 0;
        if (!uniform) {
            for (int t = 1; t < rows; t++) dpack |= uint32_t((r0 + t) * a.SR / a.R - rb0) << (4 * t);
        }
    };
    setup_tile();

    while (true) {
        // position of the next step
        int jn = j + 1;
        int64_t r0n = r0;
        int rowsn = rows;
        if (jn == iters) {
            jn = 0;
            r0n = r0 + tile_stride;
            rowsn = int(min(int64_t(T), row_end - r0n));
        }
        const bool has_next = r0n < row_end;
        uint4 nxt[T];
        if (PF && has_next) load_step<T>(nxt, a, r0n, rowsn, lane + 32 * int64_t(jn), nchunk);

        const int64_t ch = lane + 32 * int64_t(j);
        if (ch < nchunk) {
            if (uniform)
                compute_step<B, T, true>(acc, cur, a, srow0, dpack, chunk_cb[ch], ch);
            else
                compute_step<B, T, false>(acc, cur, a, srow0, dpack, chunk_cb[ch], ch);
        }
        if (j == iters - 1) {  // tile done: reduce, store, restart the sums
#pragma unroll
            for (int t = 0; t < T; t++) {
#pragma unroll
                for (int v = 0; v < B; v++) {
                    float val = warp_sum(acc[t][v]);
                    acc[t][v] = 0.0f;
                    if (t < rows) {
                        if (isnan(val)) val = f8_row_exact(a, r0 + t, v, nullptr);
                        if (lane == 0) a.y[int64_t(v) * a.R + r0 + t] = val;
                    }
                }
            }
        }
        if (!has_next) break;
        if (PF) {
#pragma unroll
            for (int t = 0; t < T; t++) cur[t] = nxt[t];
        } else {
            load_step<T>(cur, a, r0n, rowsn, lane + 32 * int64_t(jn), nchunk);
        }
        const bool new_tile = (jn == 0);
        j = jn;
        r0 = r0n;
        rows = rowsn;
        if (new_tile) setup_tile();
    }
}

// True when every 16-column chunk maps to a single scale block: the first
// column of each block b, ceil(b*C/SC), is a multiple of 16.
bool chunks_uniform(int64_t C, int64_t SC) {
    for (int64_t b = 1; b < SC; b++) {
        const int64_t start = (b * C + SC - 1) / SC;
        if (start % 16 != 0) return false;
    }
    return true;
}

template <int B, int T = (B <= 4) ? 8 : 4, bool PF = false, bool GS = true>
qmv_status launch_fast(const F8Args &a, cudaStream_t s) {
    const size_t smem = size_t(a.C >> 4) * sizeof(int);
    auto kern = f8_fast_kernel<B, T, PF, GS>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int blocks = grid_blocks(kp, 256, smem, (a.R + T - 1) / T);
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(256), smem, s, a));
}

template <int B>
qmv_status launch_general(const F8Args &a, cudaStream_t s) {
    const int blocks = grid_blocks(reinterpret_cast<const void *>(f8_general_kernel<B>), 256, 0, a.R);
    return from_cuda(launch_pdl(f8_general_kernel<B>, dim3(unsigned(blocks)), dim3(256), 0, s, a));
}

}  // namespace

qmv_status launch_f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                            int64_t SC, const float *x, int batch, float *y, cudaStream_t s) {
    F8Args a{w, scale, x, y, R, C, SR, SC};
    const bool fast = (C % 16 == 0) && (reinterpret_cast<uintptr_t>(w) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (C / 16) * 4 <= 200 * 1024 &&
                      chunks_uniform(C, SC);
    if (fast) {
        switch (batch) {
            case 1: return launch_fast<1>(a, s);
            case 2: return launch_fast<2>(a, s);
            case 3: return launch_fast<3>(a, s);
            case 4: return launch_fast<4>(a, s);
            case 5: return launch_fast<5>(a, s);
            case 6: return launch_fast<6>(a, s);
            case 7: return launch_fast<7>(a, s);
            default: return launch_fast<8>(a, s);
        }
    }
    switch (batch) {
        case 1: return launch_general<1>(a, s);
        case 2: return launch_general<2>(a, s);
        case 3: return launch_general<3>(a, s);
        case 4: return launch_general<4>(a, s);
        case 5: return launch_general<5>(a, s);
        case 6: return launch_general<6>(a, s);
        case 7: return launch_general<7>(a, s);
        default: return launch_general<8>(a, s);
    }
}

}  // namespace qmv
