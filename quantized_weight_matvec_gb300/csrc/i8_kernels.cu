// i8_kernels.cu -- int8-weight matvec with per-16 E8M0 group scales, sm_103a.
//
// Method: ds4f-disk issue #6 "attention + tokenizer + sampling", step 4 (the
// I8 matvec of simd.c: int8 weights widened, E8M0 scales per group of 16)
// and the first real tokens of step 3, which ran an I8 head over the 246k
// vocabulary.  Groups are 16 consecutive columns of a row; scale is
// [R, ceil(C/16)] row-major; code 255 is NaN, every other code 2^(e-127).
//
//   y[v][r] = sum_c w[r][c] * e8m0(scale[r][c/16]) * x[v][c]
//
// The streaming kernels walk rows like the F8 one (grid-stride tiles of T
// rows, lane l on the 16-byte chunks l, l+32, ...), so each lane's chunk is
// exactly one scale group: the chunk's 16 products are summed, then
// multiplied by the group's scale once.  Up to batch 4 the sums are exact
// int32 dot products against fixed-point limbs of x (i8_dot_kernel, below);
// otherwise int8 is widened to float32 exactly (the byte is biased to
// unsigned, permuted into the low mantissa byte of 2^23 and 2^23 + 128 is
// subtracted) and multiplied in float32.
#include <stdint.h>

#include "device_common.cuh"
#include "mma_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

struct I8Args {
    const int8_t *w;
    const uint8_t *scale;
    const float *x;
    float *y;
    int64_t R, C, SG;  // SG = ceil(C / 16) scale groups per row
    // tensor-core kernel only: when xq is set, the activations are the int8
    // codes xq [batch, C] times their per-32-column scales xd [batch, XG]
    // (i8_matvec_q8), and x is unused
    const int8_t *xq;
    const float *xd;
    int64_t XG;
};

// Activation (v, c) of an I8Args: x, or (Q8) the code times its group scale.
template <bool Q8>
__device__ __forceinline__ float act_of(const I8Args &a, int v, int64_t c) {
    if constexpr (Q8) return float(__ldg(a.xq + int64_t(v) * a.C + c)) * __ldg(a.xd + int64_t(v) * a.XG + (c >> 5));
    return __ldg(a.x + int64_t(v) * a.C + c);
}

using dev::warp_sum;

// The four int8 weights of a word as exact floats.
__device__ __forceinline__ void widen4(unsigned word, float (&f)[4]) {
    const unsigned u = word ^ 0x80808080u;
#pragma unroll
    for (int k = 0; k < 4; k++)
        f[k] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u | unsigned(k))) - 8388736.0f;
}

using dev::ld_stream;

__device__ __forceinline__ unsigned word_of(const uint4 &d, int q) {
    return q == 0 ? d.x : q == 1 ? d.y : q == 2 ? d.z : d.w;
}

// Accumulators: one float per (row, vector) at batch 1; larger batches keep
// (even column, odd column) pairs and use the packed FMA (fma.rn.f32x2).
template <int B>
struct Acc {
    typedef float2 type;
};
template <>
struct Acc<1> {
    typedef float type;
};
__device__ __forceinline__ float total(float v) { return v; }
__device__ __forceinline__ float total(float2 v) { return v.x + v.y; }
__device__ __forceinline__ void zero(float &v) { v = 0.0f; }
__device__ __forceinline__ void zero(float2 &v) { v = make_float2(0.0f, 0.0f); }

// The T weight chunks (and their scale bytes) of one step; rows past the
// tile's end and chunks past the row's end re-read in-bounds data (unused).
template <int T>
__device__ __forceinline__ void load_step(uint4 (&d)[T], unsigned (&e)[T], const I8Args &a, int64_t r0,
                                          int rows, int64_t ch, int64_t nchunk) {
    const int64_t chc = ch < nchunk ? ch : nchunk - 1;
#pragma unroll
    for (int t = 0; t < T; t++) {
        const int64_t r = r0 + (t < rows ? t : rows - 1);
        d[t] = ld_stream(a.w + r * a.C + chc * 16);
        e[t] = __ldg(a.scale + r * a.SG + chc);
    }
}

// The four int8 weights of a word as two exact float pairs, with packed
// additions of -(2^23 + 128).
__device__ __forceinline__ void widen4_pairs(unsigned word, float2 &w01, float2 &w23) {
    const unsigned u = word ^ 0x80808080u;
    const float2 k = make_float2(-8388736.0f, -8388736.0f);
    w01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u)),
                                 __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441u))), k);
    w23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442u)),
                                 __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443u))), k);
}

// acc[t][v] += e8m0(e[t]) * sum over chunk ch of w[t] * x[v].  Scalar FMAs
// at batch 1, column-paired packed FMAs otherwise.
template <int B, int T>
__device__ __forceinline__ void compute_step(typename Acc<B>::type (&acc)[T][B], const uint4 (&d)[T],
                                             const unsigned (&e)[T], const I8Args &a, int64_t ch) {
    constexpr bool SCALAR = (B == 1);
    typename Acc<B>::type part[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) zero(part[t][v]);
#pragma unroll
    for (int q = 0; q < 4; q++) {
        float4 xv[B];
#pragma unroll
        for (int v = 0; v < B; v++)
            xv[v] = __ldg(reinterpret_cast<const float4 *>(a.x + v * a.C + ch * 16 + 4 * q));
#pragma unroll
        for (int t = 0; t < T; t++) {
            if constexpr (SCALAR) {
                float f[4];
                widen4(word_of(d[t], q), f);
                part[t][0] = fmaf(f[0], xv[0].x, part[t][0]);
                part[t][0] = fmaf(f[1], xv[0].y, part[t][0]);
                part[t][0] = fmaf(f[2], xv[0].z, part[t][0]);
                part[t][0] = fmaf(f[3], xv[0].w, part[t][0]);
            } else {
                float2 w01, w23;
                widen4_pairs(word_of(d[t], q), w01, w23);
#pragma unroll
                for (int v = 0; v < B; v++) {
                    part[t][v] = __ffma2_rn(w01, make_float2(xv[v].x, xv[v].y), part[t][v]);
                    part[t][v] = __ffma2_rn(w23, make_float2(xv[v].z, xv[v].w), part[t][v]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < T; t++) {
        const float s = dev::e8m0(e[t]);
#pragma unroll
        for (int v = 0; v < B; v++) {
            if constexpr (SCALAR)
                acc[t][0] = fmaf(part[t][0], s, acc[t][0]);
            else
                acc[t][v] = __ffma2_rn(part[t][v], make_float2(s, s), acc[t][v]);
        }
    }
}

template <int B, int T>
__device__ __forceinline__ void finish_tile(typename Acc<B>::type (&acc)[T][B], const I8Args &a,
                                            int64_t r0, int rows, int lane) {
#pragma unroll
    for (int t = 0; t < T; t++) {
#pragma unroll
        for (int v = 0; v < B; v++) {
            const float val = warp_sum(total(acc[t][v]));
            zero(acc[t][v]);
            if (t < rows && lane == 0) a.y[int64_t(v) * a.R + r0 + t] = val;
        }
    }
}

// ---------------------------------------------------------------------------
// Streaming kernel (C % 16 == 0, 16-byte aligned w and x): grid-stride tiles
// of T rows, one step = the T chunks a lane owns in one 512-byte column band.
// ---------------------------------------------------------------------------
template <int B, int T>
__global__ void __launch_bounds__(256, (B == 1) ? 0 : ((B <= 4) ? 2 : 1)) i8_fast_kernel(I8Args a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nchunk = a.C >> 4;
    const int iters = int((nchunk + 31) >> 5);
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t tile_stride = nwarps * T;
    int64_t r0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * T;
    if (r0 >= a.R) return;
    int rows = int(min(int64_t(T), a.R - r0));
    typename Acc<B>::type acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) zero(acc[t][v]);
    for (int j = 0;;) {
        uint4 d[T];
        unsigned e[T];
        const int64_t ch = lane + 32 * int64_t(j);
        load_step<T>(d, e, a, r0, rows, ch, nchunk);
        if (ch < nchunk) compute_step<B, T>(acc, d, e, a, ch);
        if (++j == iters) {
            finish_tile<B, T>(acc, a, r0, rows, lane);
            r0 += tile_stride;
            if (r0 >= a.R) break;
            rows = int(min(int64_t(T), a.R - r0));
            j = 0;
        }
    }
}

// ---------------------------------------------------------------------------
// Small-matrix kernel: 2-row tiles, all NSTEP chunk steps of a tile loaded at
// once (too few rows to keep a streaming grid busy).
// ---------------------------------------------------------------------------
template <int B, int T, int NSTEP>
__global__ void __launch_bounds__(256) i8_rows_kernel(I8Args a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nchunk = a.C >> 4;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t ntiles = (a.R + T - 1) / T;
    typename Acc<B>::type acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) zero(acc[t][v]);
    for (int64_t tile = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; tile < ntiles;
         tile += nwarps) {
        const int64_t r0 = tile * T;
        const int rows = int(min(int64_t(T), a.R - r0));
        for (int64_t base = 0; base < nchunk; base += 32 * NSTEP) {
            uint4 d[NSTEP][T];
            unsigned e[NSTEP][T];
#pragma unroll
            for (int st = 0; st < NSTEP; st++)
                load_step<T>(d[st], e[st], a, r0, rows, base + lane + 32 * st, nchunk);
#pragma unroll
            for (int st = 0; st < NSTEP; st++) {
                const int64_t ch = base + lane + 32 * st;
                if (ch < nchunk) compute_step<B, T>(acc, d[st], e[st], a, ch);
            }
        }
        finish_tile<B, T>(acc, a, r0, rows, lane);
    }
}

// ---------------------------------------------------------------------------
// Split-row kernel (batch 1, 4096..16384 columns, few rows): a block of 8
// warps takes a tile of T rows and every warp a share of its columns --
// lane l of warp w reads the chunks l + 32 (w + 8 s), s < NS -- so the
// tile's T * C bytes (and their scale bytes) are requested by all 256
// threads at once, before the dependency wait, and every tile of the matrix
// is in flight in one wave.  The warps' row sums are added in shared memory
// in warp order; warp t stores row t.
// ---------------------------------------------------------------------------
constexpr int kSplitWarps = 8;

template <int T, int NS>
__global__ void __launch_bounds__(256, 4) i8_split_kernel(I8Args a) {
    static_assert(T <= kSplitWarps, "warp t stores row t");
    __shared__ float part[kSplitWarps][T];
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nchunk = a.C >> 4;
    const int64_t r0 = int64_t(blockIdx.x) * T;  // one tile per block
    const int rows = int(min(int64_t(T), a.R - r0));
    uint4 d[NS][T];
    unsigned e[NS][T];
#pragma unroll
    for (int st = 0; st < NS; st++)  // weights and their scales: before the wait
        load_step<T>(d[st], e[st], a, r0, rows, lane + 32 * (warp + kSplitWarps * st), nchunk);
    pdl_wait();
    float acc[T][1];
#pragma unroll
    for (int t = 0; t < T; t++) acc[t][0] = 0.0f;
#pragma unroll
    for (int st = 0; st < NS; st++) {
        const int64_t ch = lane + 32 * (warp + kSplitWarps * st);
        if (ch < nchunk) compute_step<1, T>(acc, d[st], e[st], a, ch);
    }
#pragma unroll
    for (int t = 0; t < T; t++) {
        const float pv = warp_sum(acc[t][0]);
        if (lane == 0) part[warp][t] = pv;
    }
    __syncthreads();
    if (warp < rows && lane == 0) {
        float val = part[0][warp];
#pragma unroll
        for (int w2 = 1; w2 < kSplitWarps; w2++) val += part[w2][warp];
        a.y[r0 + warp] = val;
    }
}

// Chunk steps per thread of the split kernel for C columns: 1, 2 or 4 (0:
// outside its range).
inline int split_steps(int64_t C) {
    const int64_t nchunk = C >> 4;
    if (nchunk < 32 * kSplitWarps) return 0;
    for (int ns = 1; ns <= 4; ns *= 2)
        if (nchunk <= int64_t(32) * kSplitWarps * ns) return ns;
    return 0;
}

template <int T, int NS>
qmv_status launch_i8_split_t(const I8Args &a, cudaStream_t s, bool &taken) {
    const void *kp = reinterpret_cast<const void *>(i8_split_kernel<T, NS>);
    const int64_t tiles = (a.R + T - 1) / T;
    taken = tiles <= int64_t(occupancy(kp, 256, 0)) * sm_count();  // every tile resident
    if (!taken) return QMV_OK;
    return from_cuda(launch_pdl(i8_split_kernel<T, NS>, dim3(unsigned(tiles)), dim3(256), 0, s, a));
}

// Runs the split kernel when it takes the call (batch 1, C % 16 == 0 and
// aligned pointers checked by the caller); `taken` says whether it did.
qmv_status launch_i8_split(const I8Args &a, cudaStream_t s, bool &taken) {
    switch (split_steps(a.C)) {
        case 1: return launch_i8_split_t<8, 1>(a, s, taken);
        case 2: return launch_i8_split_t<4, 2>(a, s, taken);
        case 4: return launch_i8_split_t<2, 4>(a, s, taken);
        default: taken = false; return QMV_OK;
    }
}

// ---------------------------------------------------------------------------
// General kernel: any C and alignment.  One warp per row, one element per
// lane step: (w * scale) * x in a float32 FMA.
// ---------------------------------------------------------------------------
template <int B>
__global__ void __launch_bounds__(256) i8_general_kernel(I8Args a) {
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
            const float ws = float(__ldg(wr + c)) * dev::e8m0(__ldg(sr + (c >> 4)));
#pragma unroll
            for (int v = 0; v < B; v++) acc[v] = fmaf(ws, __ldg(a.x + v * a.C + c), acc[v]);
        }
#pragma unroll
        for (int v = 0; v < B; v++) {
            const float val = warp_sum(acc[v]);
            if (lane == 0) a.y[int64_t(v) * a.R + r] = val;
        }
    }
}

// ---------------------------------------------------------------------------
// Integer-dot kernel (C % 16 == 0, 16-byte aligned w and x).
//
// Each 16-column group of x is written once per block as fixed-point
// integers relative to the group's largest finite |x|: with m in
// [2^(k-1), 2^k) and E = min(29 - k, 149), x_int = rint(x * 2^E) has
// |x_int| <= 2^29, and x = (x_int + err) * 2^-E with |err| <= 1/2, i.e. an
// absolute error of at most 2^-30 * m per element.  x_int is split into two
// signed 16-bit limbs, x_int = hi * 2^15 + lo (lo in [-2^14, 2^14)), so that
// dp2a (two int16 x int8 products and an add per instruction) forms the
// group's sums sum_c w_c * hi_c and sum_c w_c * lo_c exactly in int32
// (each at most 16 * 128 * (2^14 + 1) in magnitude).  The group result is
// (float(sum_hi) * 2^15 + float(sum_lo)) * 2^-E * e8m0(scale), accumulated in
// float32.  This is the integer-dot scheme of the Mnemonic page ("In the
// browser": int8 weights against activations scaled per group and widened
// to int16, exact int32 sums, then floats times the group scale), with
// 31-bit instead of 8-bit activations so that the result stays within the
// float32-accumulation tolerance.  A group holding Inf or NaN is flagged
// (its 2^-E is stored as NaN) and evaluated in float32 from x directly.
// ---------------------------------------------------------------------------

// Shared-memory layout, per vector v and step j (32 chunks = 512 columns):
//   limbs[v][j][part][lane]  uint4: part 0/1 = lo limbs of columns 0-7 / 8-15
//                            of the lane's chunk, part 2/3 = hi limbs
//   xs[v][j][lane]           float: 2^-E of the chunk's group (NaN: flagged)
__device__ __forceinline__ unsigned pack_s16(int a, int b) {
    return (unsigned(a) & 0xffffu) | (unsigned(b) << 16);
}

__device__ void prep_x_limbs(const I8Args &a, int B, int nj, uint4 *limbs, float *xs) {
    const int64_t nchunk = a.C >> 4;
    const int jobs = B * nj * 32;
    for (int job = threadIdx.x; job < jobs; job += blockDim.x) {
        const int v = job / (nj * 32), rem = job - v * nj * 32;
        const int j = rem >> 5, lane = rem & 31;
        const int64_t ch = int64_t(j) * 32 + lane;
        uint4 *out = limbs + (int64_t(v * nj + j) * 4) * 32 + lane;
        float sx = 0.0f;
        unsigned lw[8] = {0, 0, 0, 0, 0, 0, 0, 0}, hw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (ch < nchunk) {
            const float4 *xp = reinterpret_cast<const float4 *>(a.x + int64_t(v) * a.C + ch * 16);
            float xv[16];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 t = __ldg(xp + q);
                xv[4 * q] = t.x;
                xv[4 * q + 1] = t.y;
                xv[4 * q + 2] = t.z;
                xv[4 * q + 3] = t.w;
            }
            float m = 0.0f;
            bool finite = true;
#pragma unroll
            for (int c = 0; c < 16; c++) {
                finite = finite && isfinite(xv[c]);
                m = fmaxf(m, fabsf(xv[c]));
            }
            if (!finite) {
                sx = __uint_as_float(0x7fc00000u);
            } else {
                int k = 0;
                frexpf(m, &k);
                const int E = m == 0.0f ? 0 : min(29 - k, 149);
                sx = scalbnf(1.0f, -E);
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    int xi0 = __float2int_rn(scalbnf(xv[c], E));
                    int xi1 = __float2int_rn(scalbnf(xv[c + 1], E));
                    const int lo0 = ((xi0 + 0x4000) & 0x7fff) - 0x4000;
                    const int lo1 = ((xi1 + 0x4000) & 0x7fff) - 0x4000;
                    lw[c >> 1] = pack_s16(lo0, lo1);
                    hw[c >> 1] = pack_s16((xi0 - lo0) >> 15, (xi1 - lo1) >> 15);
                }
            }
        }
        out[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        out[32] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        out[64] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        out[96] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        xs[int64_t(v * nj + j) * 32 + lane] = sx;
    }
}

__device__ __forceinline__ unsigned limb_word(const uint4 &p0, const uint4 &p1, int i) {
    const uint4 &p = i < 4 ? p0 : p1;
    const int k = i & 3;
    return k == 0 ? p.x : k == 1 ? p.y : k == 2 ? p.z : p.w;
}

template <int B, int T>
__global__ void __launch_bounds__(256) i8_dot_kernel(I8Args a, int nj) {
    extern __shared__ uint4 dsm[];
    uint4 *limbs = dsm;
    float *xs = reinterpret_cast<float *>(dsm + int64_t(B) * nj * 128);
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nchunk = a.C >> 4;
    const int iters = int((nchunk + 31) >> 5);
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t tile_stride = nwarps * T;
    int64_t r0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * T;
    int rows = int(min(int64_t(T), a.R - max(r0, int64_t(0))));
    // first step's weights in flight before the dependency wait (they never
    // depend on the preceding kernel) and while x is converted
    uint4 d[T];
    unsigned e[T];
    if (r0 < a.R) load_step<T>(d, e, a, r0, rows, lane, nchunk);
    pdl_wait();
    prep_x_limbs(a, B, nj, limbs, xs);
    __syncthreads();
    if (r0 >= a.R) return;
    float acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) acc[t][v] = 0.0f;
    for (int j = 0;;) {
        const int64_t ch = lane + 32 * int64_t(j);
        if (ch < nchunk) {
            float sw[T];
#pragma unroll
            for (int t = 0; t < T; t++) sw[t] = dev::e8m0(e[t]);
#pragma unroll
            for (int v = 0; v < B; v++) {
                const uint4 *lp = limbs + (int64_t(v * nj + j) * 4) * 32 + lane;
                const uint4 l0 = lp[0], l1 = lp[32], h0 = lp[64], h1 = lp[96];
                const float sx = xs[int64_t(v * nj + j) * 32 + lane];
                if (isnan(sx)) {
                    // group with Inf/NaN in x: float32 products from x itself
                    const float *xv = a.x + int64_t(v) * a.C + ch * 16;
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        float part = 0.0f;
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            float f[4];
                            widen4(word_of(d[t], q), f);
#pragma unroll
                            for (int k = 0; k < 4; k++) part = fmaf(f[k], __ldg(xv + 4 * q + k), part);
                        }
                        acc[t][v] = fmaf(part, sw[t], acc[t][v]);
                    }
                    continue;
                }
#pragma unroll
                for (int t = 0; t < T; t++) {
                    int sl = 0, sh = 0;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int wq = int(word_of(d[t], q));
                        sl = __dp2a_lo(int(limb_word(l0, l1, 2 * q)), wq, sl);
                        sl = __dp2a_hi(int(limb_word(l0, l1, 2 * q + 1)), wq, sl);
                        sh = __dp2a_lo(int(limb_word(h0, h1, 2 * q)), wq, sh);
                        sh = __dp2a_hi(int(limb_word(h0, h1, 2 * q + 1)), wq, sh);
                    }
                    const float g = fmaf(__int2float_rn(sh), 32768.0f, __int2float_rn(sl));
                    acc[t][v] = fmaf(g * sx, sw[t], acc[t][v]);
                }
            }
        }
        if (++j == iters) {
#pragma unroll
            for (int t = 0; t < T; t++) {
#pragma unroll
                for (int v = 0; v < B; v++) {
                    const float val = warp_sum(acc[t][v]);
                    acc[t][v] = 0.0f;
                    if (t < rows && lane == 0) a.y[int64_t(v) * a.R + r0 + t] = val;
                }
            }
            r0 += tile_stride;
            if (r0 >= a.R) break;
            rows = int(min(int64_t(T), a.R - r0));
            j = 0;
        }
        load_step<T>(d, e, a, r0, rows, lane + 32 * int64_t(j), nchunk);
    }
}

// Shared memory of i8_dot_kernel for B vectors of C columns.
inline size_t dot_smem(int B, int64_t C) {
    const int64_t nj = ((C >> 4) + 31) >> 5;
    return size_t(B) * size_t(nj) * (128 * 16 + 32 * 4);
}

template <int B, int T>
qmv_status launch_i8_dot(const I8Args &a, cudaStream_t s) {
    const int nj = int(((a.C >> 4) + 31) >> 5);
    const size_t smem = dot_smem(B, a.C);
    const void *kp = reinterpret_cast<const void *>(i8_dot_kernel<B, T>);
    if (smem > 48 * 1024 && !allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int blocks = grid_blocks(kp, 256, smem, (a.R + T - 1) / T);
    return from_cuda(launch_pdl(i8_dot_kernel<B, T>, dim3(unsigned(blocks)), dim3(256), smem, s, a, nj));
}

// Largest shared memory the integer-dot kernel may take (x limbs of all
// vectors); wider rows run on the float kernel.
constexpr size_t kDotSmemMax = 160 * 1024;

// ---------------------------------------------------------------------------
// Batch 2..8: the multiply-accumulate on the tensor cores (mma.sync m16n8k16,
// f16 operands, float32 accumulation), in the staged layout of the F8 kernel
// (mma_device.cuh): weights copied into a three-deep shared-memory ring with
// cp.async, B fragments (x split into f16 hi + lo per 64-column block) in
// registers, a fixed-order tile epilogue.
//
// In that layout lane (g, t) holds, for rows g and g+8, the 16 bytes at
// column 64*kb + 16*t: exactly one scale group.  So the group scale is folded
// into the weights as they are decoded: the byte is biased to unsigned and
// placed in the low mantissa byte of 1024 (f16 0x6400), and one f16 fma by
// (s, s) with addend -1152 s gives w * s -- the exact product, rounded once,
// hence exact whenever w * s is an f16: for every scale 2^-24 <= s <= 2^5
// (codes 103..132).  The mma then mixes groups freely.  A row with any group
// scale outside that range gets NaN weights, so the epilogue recomputes it
// by the exact per-element path (as it does for non-finite x and the NaN
// scale code 255).
// ---------------------------------------------------------------------------

// Exact per-element value of output (r, v) (warp-collective).
template <bool Q8>
__device__ float i8_row_exact(const I8Args &a, int64_t r, int v) {
    const int lane = threadIdx.x & 31;
    const int8_t *wr = a.w + r * a.C;
    const uint8_t *sr = a.scale + r * a.SG;
    float acc = 0.0f;
    for (int64_t c = lane; c < a.C; c += 32) {
        const float ws = float(__ldg(wr + c)) * dev::e8m0(__ldg(sr + (c >> 4)));
        acc = fmaf(ws, act_of<Q8>(a, v, c), acc);
    }
    return warp_sum(acc);
}

template <bool Q8>
struct I8Exact {
    const I8Args &a;
    __device__ __forceinline__ float operator()(int64_t r, int v) const { return i8_row_exact<Q8>(a, r, v); }
};

__device__ __forceinline__ bool no_better(float, int64_t, float, int64_t) { return false; }

// E8M0 code e -> f16x2 (s, s) and (-1152 s, -1152 s); `ok` false (and NaN
// pairs) outside 103..132, where w * s is not always an f16.
__device__ __forceinline__ void i8_fold(unsigned e, uint32_t &s2, uint32_t &c2, bool &ok) {
    ok = (e - 103u) <= 29u;
    const uint32_t sb = e >= 113u ? (e - 112u) << 10 : 1u << ((e - 103u) & 31u);
    const uint32_t cb = 0x8000u | (((e - 102u) & 31u) << 10) | 0x080u;
    s2 = ok ? (sb | (sb << 16)) : 0x7e007e00u;
    c2 = ok ? (cb | (cb << 16)) : 0x7e007e00u;
}

// Four int8 weights of a word times their group scale, as two f16 pairs
// (bytes 0-1 -> lo, bytes 2-3 -> hi).
__device__ __forceinline__ void i8x4_fold(uint32_t w, uint32_t s2, uint32_t c2, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t m01 = __byte_perm(u, 0x64646464u, 0x4140u), m23 = __byte_perm(u, 0x64646464u, 0x4342u);
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(m01), "r"(s2), "r"(c2));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(hi) : "r"(m23), "r"(s2), "r"(c2));
}

template <int NJ, int NK, bool Q8, bool EARLY>
__global__ void __launch_bounds__(512, 1) i8_mma_staged_kernel(I8Args a, int batch) {
    constexpr bool kEarly = NJ == 1 || EARLY;  // first tiles issued before the dependency wait
    extern __shared__ __align__(16) unsigned char st_smem[];
    using namespace mma;
    constexpr int NCH = 4 * NK;          // 16-byte chunks per row and warp
    constexpr int SLOT = 16 * NCH * 16;  // bytes per warp and stage
    const int NW = blockDim.x >> 5;      // warp w owns column blocks [w NK, w NK + NK)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int kb_lo = warp * NK;
    const uint32_t ring = uint32_t(__cvta_generic_to_shared(st_smem)) + uint32_t(warp * kRing * SLOT);
    const uint4 *ring_g = reinterpret_cast<const uint4 *>(st_smem + size_t(warp) * kRing * SLOT);
    float *red = reinterpret_cast<float *>(st_smem + size_t(NW) * kRing * SLOT);
    const uint8_t *w8 = reinterpret_cast<const uint8_t *>(a.w);

    if (kEarly) pdl_trigger();

    const int64_t ntiles = (a.R + 15) >> 4;
    const int64_t gstride = gridDim.x;
    float best_v = 0.0f;
    int64_t best_i = 0;
    // E8M0 codes of the lane's groups (4 (kb_lo + k) + t) of rows g and g+8
    auto load_scales = [&](int64_t tl, unsigned (&sa)[NK], unsigned (&sb)[NK]) {
        const int64_t ra = min(tl * 16 + g, a.R - 1), rb = min(tl * 16 + g + 8, a.R - 1);
        const uint8_t *pa = a.scale + ra * a.SG + 4 * kb_lo + t, *pb = a.scale + rb * a.SG + 4 * kb_lo + t;
#pragma unroll
        for (int k = 0; k < NK; k++) {
            sa[k] = __ldg(pa + 4 * k);
            sb[k] = __ldg(pb + 4 * k);
        }
    };
    // the first kRing - 1 tiles of weights and the first tile's scale codes
    // go out before the dependency wait (they never depend on the preceding
    // kernel); at batch 5-8 (NJ = 2), where the kernel sits at its register
    // limit, only for matrices of a few tiles per block (EARLY: 4096 x 4096
    // at batch 8 12.6 -> 11.3 us, while on the head 221 -> 246 us), else
    // after it
    unsigned sa[NK], sb[NK];
    auto issue_first = [&]() {
        if (int64_t(blockIdx.x) < ntiles) {  // block-uniform
#pragma unroll
            for (int st = 0; st < kRing - 1; st++) {
                const int64_t tl = blockIdx.x + st * gstride;
                if (tl < ntiles) issue_tile<NK>(ring + uint32_t(st * SLOT), w8, a.R, a.C, tl, kb_lo, lane);
                cp_async_commit();
            }
            load_scales(blockIdx.x, sa, sb);
        }
    };
    if (kEarly) issue_first();
    pdl_wait();
    if (!kEarly) {
        pdl_trigger();
        issue_first();
    }
    if (int64_t(blockIdx.x) < ntiles) {  // block-uniform
        StagedB<NJ> B;
        if constexpr (Q8) {
            // q * d of the chunk's 32-column group (16-byte aligned codes)
            auto load16 = [&](int v, int64_t c0, float (&xs)[16]) {
                const uint4 qv = __ldg(reinterpret_cast<const uint4 *>(a.xq + int64_t(v) * a.C + c0));
                const float dv = __ldg(a.xd + int64_t(v) * a.XG + (c0 >> 5));
                const unsigned wq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int e = 0; e < 16; e++) xs[e] = float(int8_t(wq[e >> 2] >> (8 * (e & 3)))) * dv;
            };
            build_b_from<NJ>(B, load16, batch, kb_lo, NK, lane);
        } else {
            build_b<NJ>(B, a.x, a.C, batch, kb_lo, NK, lane);
        }

        float tot[NJ][2];
#pragma unroll
        for (int j = 0; j < NJ; j++) tot[j][0] = tot[j][1] = 0.0f;
        int buf = 0, slot = 0;
        for (int64_t tl = blockIdx.x; tl < ntiles; tl += gstride) {
            {
                const int64_t tn = tl + (kRing - 1) * gstride;
                int sn = slot + kRing - 1;
                if (sn >= kRing) sn -= kRing;
                if (tn < ntiles) issue_tile<NK>(ring + uint32_t(sn * SLOT), w8, a.R, a.C, tn, kb_lo, lane);
                cp_async_commit();
            }
            unsigned san[NK], sbn[NK];
            if (tl + gstride < ntiles) {
                load_scales(tl + gstride, san, sbn);
            } else {
#pragma unroll
                for (int k = 0; k < NK; k++) san[k] = sbn[k] = 127u;
            }
            cp_async_wait<kRing - 1>();  // this lane's copies of the tile have landed
            __syncwarp();                // ... and every other lane's
            const uint4 *src = ring_g + slot * (SLOT / 16);
#pragma unroll
            for (int k = 0; k < NK; k++) {
                const uint4 wa4 = row_chunk<NK>(src, g, 4 * k + t);
                const uint4 wb4 = row_chunk<NK>(src, g + 8, 4 * k + t);
                uint32_t sa2, ca2, sb2, cb2;
                bool oka, okb;
                i8_fold(sa[k], sa2, ca2, oka);
                i8_fold(sb[k], sb2, cb2, okb);
                constexpr int NA = NJ == 1 ? 2 : 1;
                float acc[NA][NJ][4];
#pragma unroll
                for (int q = 0; q < NA; q++)
#pragma unroll
                    for (int j = 0; j < NJ; j++) acc[q][j][0] = acc[q][j][1] = acc[q][j][2] = acc[q][j][3] = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    uint32_t a0, a2, a1, a3;
                    i8x4_fold(word_of(wa4, i), sa2, ca2, a0, a2);
                    i8x4_fold(word_of(wb4, i), sb2, cb2, a1, a3);
#pragma unroll
                    for (int j = 0; j < NJ; j++)
                        mma_16816(acc[i % NA][j], a0, a1, a2, a3, B.b[k][i][j][0], B.b[k][i][j][1]);
                }
#pragma unroll
                for (int j = 0; j < NJ; j++) {
                    const float f = B.f[k][j];
                    float ha = acc[0][j][0] + acc[0][j][1], hb = acc[0][j][2] + acc[0][j][3];
                    if (NA == 2) {
                        ha += acc[NA - 1][j][0] + acc[NA - 1][j][1];
                        hb += acc[NA - 1][j][2] + acc[NA - 1][j][3];
                    }
                    tot[j][0] = fmaf(ha, f, tot[j][0]);
                    tot[j][1] = fmaf(hb, f, tot[j][1]);
                }
            }
            tile_epilogue<NJ, false>(tot, red, buf, NW, batch, a.R, a.y, tl * 16, best_v, best_i, I8Exact<Q8>{a},
                                     no_better);
            buf ^= 1;
            if (++slot == kRing) slot = 0;
#pragma unroll
            for (int k = 0; k < NK; k++) {
                sa[k] = san[k];
                sb[k] = sbn[k];
            }
        }
        cp_async_wait<0>();  // (only empty groups can remain)
    }
}

// Batch 5-8 matrices of at most this many 16-row tiles per block issue their
// first tiles before the dependency wait (EARLY).
constexpr int64_t kEarlyTilesPerBlock = 8;

template <int NJ, int NK, bool Q8 = false, bool EARLY = false>
qmv_status launch_i8_mma(const I8Args &a, int batch, cudaStream_t s) {
    const int NW = int(a.C / 64 / NK);
    const size_t smem = mma::staged_smem_bytes(NW, NK, NJ, 0);
    auto kern = i8_mma_staged_kernel<NJ, NK, Q8, EARLY>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int64_t ntiles = (a.R + 15) / 16;
    int64_t blocks = int64_t(occupancy(kp, 32 * NW, smem)) * sm_count();
    if (blocks > ntiles) blocks = ntiles;
    if constexpr (NJ == 2 && !EARLY) {
        if (ntiles <= kEarlyTilesPerBlock * blocks) return launch_i8_mma<NJ, NK, Q8, true>(a, batch, s);
    }
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(32 * NW), smem, s, a, batch));
}

template <int NJ, bool Q8 = false>
qmv_status launch_i8_mma_any(const I8Args &a, int batch, int nk, cudaStream_t s) {
    switch (nk) {
        case 4: return launch_i8_mma<NJ, 4, Q8>(a, batch, s);
        case 2: return launch_i8_mma<NJ, 2, Q8>(a, batch, s);
        default: return launch_i8_mma<NJ, 1, Q8>(a, batch, s);
    }
}

template <int B>
qmv_status launch_i8(const I8Args &a, cudaStream_t s) {
    const bool fast = (a.C % 16 == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(a.x) % 16 == 0);
    if (!fast) {
        const void *kp = reinterpret_cast<const void *>(i8_general_kernel<B>);
        const int blocks = grid_blocks(kp, 256, 0, a.R);
        return from_cuda(launch_pdl(i8_general_kernel<B>, dim3(unsigned(blocks)), dim3(256), 0, s, a));
    }
    // Batch 2..8 on the tensor cores (C % 64 == 0, 256 <= C <= 4096)
    if (B >= 2 && a.C >= 256) {
        const int nk = mma::staged_nk(a.C, B);
        if (nk) return launch_i8_mma_any<(B + 3) / 4>(a, B, nk, s);
    }
    // Batch 1, few rows of 4096..16384 columns: one wave, columns split over warps
    if (B == 1) {
        bool taken = false;
        const qmv_status st = launch_i8_split(a, s, taken);
        if (taken) return st;
    }
    // Too few tiles to keep a streaming grid busy: the small-matrix kernel
    // (at 4096 rows it also beats converting x in every block).
    constexpr int T = 4;
    const void *kp = reinterpret_cast<const void *>(i8_fast_kernel<B, T>);
    const int64_t capacity = int64_t(occupancy(kp, 256, 0)) * sm_count() * 8;
    if ((a.R + T - 1) / T < 4 * capacity) {
        constexpr int TS = 2, NSTEP = (B <= 2) ? 8 : 4;
        const void *rp = reinterpret_cast<const void *>(i8_rows_kernel<B, TS, NSTEP>);
        const int blocks = grid_blocks(rp, 256, 0, (a.R + TS - 1) / TS);
        return from_cuda(launch_pdl(i8_rows_kernel<B, TS, NSTEP>, dim3(unsigned(blocks)), dim3(256), 0, s, a));
    }
    // Integer dot products up to batch 4: one dp2a per weight and vector is
    // cheaper than widening every weight to float, until the dp2a rate
    // (half the FMA rate) runs out at larger batches.  Tile heights from a
    // sweep on the 245760 x 4096 head: 6 rows at batch 1-2, 4 at 3-4.
    if (B <= 4 && dot_smem(B, a.C) <= kDotSmemMax) return launch_i8_dot<B, (B <= 2) ? 6 : 4>(a, s);
    const int blocks = grid_blocks(kp, 256, 0, (a.R + T - 1) / T);
    return from_cuda(launch_pdl(i8_fast_kernel<B, T>, dim3(unsigned(blocks)), dim3(256), 0, s, a));
}

}  // namespace

bool launch_i8_matvec_q8_mma(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale, const int8_t *xq,
                             const float *xd, int batch, float *y, cudaStream_t s, qmv_status &st) {
    if (batch < 2 || C < 256 || (reinterpret_cast<uintptr_t>(w) % 16) != 0 ||
        (reinterpret_cast<uintptr_t>(xq) % 16) != 0)
        return false;
    const int nk = mma::staged_nk(C, batch);
    if (!nk) return false;
    I8Args a{w, scale, nullptr, y, R, C, (C + 15) / 16, xq, xd, (C + 31) / 32};
    st = (batch <= 4) ? launch_i8_mma_any<1, true>(a, batch, nk, s) : launch_i8_mma_any<2, true>(a, batch, nk, s);
    return true;
}

qmv_status launch_i8_matvec(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale, const float *x,
                            int batch, float *y, cudaStream_t s) {
    I8Args a{w, scale, x, y, R, C, (C + 15) / 16};
    switch (batch) {
        case 1: return launch_i8<1>(a, s);
        case 2: return launch_i8<2>(a, s);
        case 3: return launch_i8<3>(a, s);
        case 4: return launch_i8<4>(a, s);
        case 5: return launch_i8<5>(a, s);
        case 6: return launch_i8<6>(a, s);
        case 7: return launch_i8<7>(a, s);
        default: return launch_i8<8>(a, s);
    }
}

}  // namespace qmv
