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

#include "mma_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

using mma::cp_async_commit;
using mma::cp_async_wait;
using mma::kRing;
using mma::mma_16816;
using mma::split_block;

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
    ArgBest *ws;  // argmax variant: [gridDim.x, B] partial results
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
template <int B, bool AM>
__global__ void __launch_bounds__(256) f8_general_kernel(F8Args a) {
    __shared__ float lut[256];
    lut[threadIdx.x] = e4m3_exact(threadIdx.x);
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    WarpBest<B> best;
    best.init();
    for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < a.R; r += nwarps) {
#pragma unroll
        for (int v = 0; v < B; v++) {
            const float val = f8_row_exact(a, r, v, lut);
            if (AM) best.offer(v, val, r);
            if (lane == 0 && (!AM || a.y)) a.y[int64_t(v) * a.R + r] = val;
        }
    }
    if (AM) block_best_store<B>(best, a.ws);
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

// Accumulators: batch 1 keeps one float per row and folds the chunk's scale
// into x (one multiply shared by the T rows); larger batches keep an
// (even column, odd column) pair per row and vector, fold the scale into the
// decoded weight pair (one packed multiply shared by the B vectors) and use
// one packed FMA (fma.rn.f32x2) per weight pair and vector.
template <int B>
struct AccOf {
    typedef float2 type;
};
template <>
struct AccOf<1> {
    typedef float type;
};
__device__ __forceinline__ float acc_total(float v) { return v; }
__device__ __forceinline__ float acc_total(float2 v) { return v.x + v.y; }
__device__ __forceinline__ void acc_zero(float &v) { v = 0.0f; }
__device__ __forceinline__ void acc_zero(float2 &v) { v = make_float2(0.0f, 0.0f); }

__device__ __forceinline__ void decode_pairs(unsigned word, float2 &w01, float2 &w23) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(word & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(word >> 16), __NV_E4M3);
    w01 = __half22float2(__half2(lo));
    w23 = __half22float2(__half2(hi));
}

// acc[t][v] += sum over the 16 columns of chunk ch of w[t] * s_t * x[v].
// UNIFORM: every row of the tile uses the scale row srow0; otherwise row t
// uses srow0 + ((dpack >> 4t) & 15) * SC.
template <int B, int T, bool UNIFORM>
__device__ __forceinline__ void compute_step(typename AccOf<B>::type (&acc)[T][B], const uint4 (&d)[T],
                                             const F8Args &a, const uint8_t *srow0, uint32_t dpack, int cb,
                                             int64_t ch) {
    // scale of row t for this chunk
    const float s0 = e8m0_value(__ldg(srow0 + cb));
    auto scale_of = [&](int t) -> float {
        return UNIFORM ? s0 : e8m0_value(__ldg(srow0 + int64_t((dpack >> (4 * t)) & 15u) * a.SC + cb));
    };
#pragma unroll
    for (int q = 0; q < 4; q++) {
        float4 xv[B];
#pragma unroll
        for (int v = 0; v < B; v++)
            xv[v] = __ldg(reinterpret_cast<const float4 *>(a.x + v * a.C + ch * 16 + 4 * q));
        if constexpr (B == 1) {
            float4 xs = make_float4(xv[0].x * s0, xv[0].y * s0, xv[0].z * s0, xv[0].w * s0);
#pragma unroll
            for (int t = 0; t < T; t++) {
                if (!UNIFORM) {
                    const float st = scale_of(t);
                    xs = make_float4(xv[0].x * st, xv[0].y * st, xv[0].z * st, xv[0].w * st);
                }
                float2 w01, w23;
                decode_pairs(word_of(d[t], q), w01, w23);
                acc[t][0] = fmaf(w01.x, xs.x, acc[t][0]);
                acc[t][0] = fmaf(w01.y, xs.y, acc[t][0]);
                acc[t][0] = fmaf(w23.x, xs.z, acc[t][0]);
                acc[t][0] = fmaf(w23.y, xs.w, acc[t][0]);
            }
        } else {
#pragma unroll
            for (int t = 0; t < T; t++) {
                float2 w01, w23;
                decode_pairs(word_of(d[t], q), w01, w23);
                const float st = scale_of(t);
                const float2 ss = make_float2(st, st);
                w01 = __fmul2_rn(w01, ss);
                w23 = __fmul2_rn(w23, ss);
#pragma unroll
                for (int v = 0; v < B; v++) {
                    acc[t][v] = __ffma2_rn(w01, make_float2(xv[v].x, xv[v].y), acc[t][v]);
                    acc[t][v] = __ffma2_rn(w23, make_float2(xv[v].z, xv[v].w), acc[t][v]);
                }
            }
        }
    }
}

// Tile epilogue: reduce each row's sums across the warp (fixed order), fall
// back to the exact per-element evaluation for rows that came out NaN, store.
template <int B, int T, bool AM>
__device__ __forceinline__ void finish_tile(typename AccOf<B>::type (&acc)[T][B], const F8Args &a, int64_t r0,
                                            int rows, int lane, WarpBest<B> &best) {
#pragma unroll
    for (int t = 0; t < T; t++) {
#pragma unroll
        for (int v = 0; v < B; v++) {
            float val = warp_sum(acc_total(acc[t][v]));
            acc_zero(acc[t][v]);
            if (t < rows) {
                if (isnan(val)) val = f8_row_exact(a, r0 + t, v, nullptr);
                if (AM) best.offer(v, val, r0 + t);
                if (lane == 0 && (!AM || a.y)) a.y[int64_t(v) * a.R + r0 + t] = val;
            }
        }
    }
}

// Scale rows of a tile: srow0 for its first row and, when the tile spans
// several scale rows, 4-bit per-row offsets (rows of one tile span at most
// T + 1 scale rows since SR <= R).
template <int T>
__device__ __forceinline__ bool setup_scale(const F8Args &a, int64_t r0, int rows, const uint8_t *&srow0,
                                            uint32_t &dpack) {
    static_assert(T <= 8, "per-row scale offsets are packed in 4 bits");
    const int64_t rb0 = r0 * a.SR / a.R, rb1 = (r0 + rows - 1) * a.SR / a.R;
    srow0 = a.scale + rb0 * a.SC;
    dpack = 0;
    if (rb0 == rb1) return true;
    for (int t = 1; t < rows; t++) dpack |= uint32_t((r0 + t) * a.SR / a.R - rb0) << (4 * t);
    return false;
}

// Resident blocks per SM the register budget is sized for: batch 1 streams
// best at 3 blocks (the plain variant fits there on its own; the argmax
// variant is held to it), batches up to 4 at 2, larger batches at 1.
template <int B, bool AM>
struct FastMinBlocks {
    static constexpr int value = (B == 1) ? (AM ? 3 : 0) : (B <= 4 ? 2 : 1);
};

template <int B, int T, bool PF, bool GS, bool AM>
__global__ void __launch_bounds__(256, FastMinBlocks<B, AM>::value) f8_fast_kernel(F8Args a) {
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
    WarpBest<B> best;
    best.init();
    if (r0 < row_end) {  // (no early return: the argmax epilogue has a barrier)
    const int iters = int((nchunk + 31) >> 5);

    int rows = int(min(int64_t(T), row_end - r0));
    int j = 0;
    uint4 cur[T];
    load_step<T>(cur, a, r0, rows, lane, nchunk);

    typename AccOf<B>::type acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) acc_zero(acc[t][v]);

    const uint8_t *srow0 = a.scale;
    uint32_t dpack = 0;
    bool uniform = true;
    auto setup_tile = [&]() { uniform = setup_scale<T>(a, r0, rows, srow0, dpack); };
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
        if (j == iters - 1) finish_tile<B, T, AM>(acc, a, r0, rows, lane, best);  // tile done
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
    if (AM) block_best_store<B>(best, a.ws);
}

// ---------------------------------------------------------------------------
// Small-matrix kernel: when the matrix has too few rows to give every warp of
// a full grid several tiles, each warp takes tiles of T rows and loads all
// NSTEP chunk steps of them at once (NSTEP * 512 bytes per row in flight),
// so the whole matrix is requested in about one wave instead of NSTEP
// dependent round trips per warp.  Same arithmetic and order as the fast
// kernel.
// ---------------------------------------------------------------------------
template <int B, int T, int NSTEP, bool AM>
__global__ void __launch_bounds__(256) f8_rows_kernel(F8Args a) {
    extern __shared__ int chunk_cb[];
    const int64_t nchunk = a.C >> 4;
    for (int64_t ch = threadIdx.x; ch < nchunk; ch += blockDim.x)
        chunk_cb[ch] = int((ch * 16 * a.SC) / a.C);
    pdl_wait();
    pdl_trigger();
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t ntiles = (a.R + T - 1) / T;
    typename AccOf<B>::type acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) acc_zero(acc[t][v]);

    WarpBest<B> best;
    best.init();
    for (int64_t tile = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; tile < ntiles;
         tile += nwarps) {
        const int64_t r0 = tile * T;
        const int rows = int(min(int64_t(T), a.R - r0));
        const uint8_t *srow0;
        uint32_t dpack;
        const bool uniform = setup_scale<T>(a, r0, rows, srow0, dpack);
        for (int64_t base = 0; base < nchunk; base += 32 * NSTEP) {
            uint4 d[NSTEP][T];
#pragma unroll
            for (int st = 0; st < NSTEP; st++) load_step<T>(d[st], a, r0, rows, base + lane + 32 * st, nchunk);
#pragma unroll
            for (int st = 0; st < NSTEP; st++) {
                const int64_t ch = base + lane + 32 * st;
                if (ch < nchunk) {
                    if (uniform)
                        compute_step<B, T, true>(acc, d[st], a, srow0, dpack, chunk_cb[ch], ch);
                    else
                        compute_step<B, T, false>(acc, d[st], a, srow0, dpack, chunk_cb[ch], ch);
                }
            }
        }
        finish_tile<B, T, AM>(acc, a, r0, rows, lane, best);
    }
    if (AM) block_best_store<B>(best, a.ws);
}

// ---------------------------------------------------------------------------
// Batch 2..8: the multiply-accumulate on the tensor cores.
//
// At batch > 1 every weight meets B activations, and on the CUDA cores that
// is B FMAs per weight plus a re-read of x per row tile: the float kernel
// above stops well short of the weight stream (L1 data pipe and issue
// bound).  Here each warp hands the products to mma.sync m16n8k16 (f16
// operands, float32 accumulation), which takes a 16-row x 16-column block of
// decoded weights against 8 activation columns per instruction.
//
// Operands.  A = 16 weight rows, decoded in registers with
// cvt.rn.f16x2.e4m3x2 (exact: every finite E4M3 value is an f16).  B = the
// activations, split so the f16 operands lose nothing that matters: per
// vector v and 64-column block kb, with m the largest finite |x| there and
// E = 14 - floor(log2 m) (at most 127), x * 2^E = hi + lo with hi = f16(x * 2^E)
// and lo = f16(x * 2^E - hi), so hi + lo carries x to 2^-22 relative (2^-25
// absolute, in units where m is ~2^14, once lo is an f16 subnormal).  The 8
// columns of one mma are (vector, hi|lo) pairs of 4 vectors; batches 5..8 take
// a second mma on the same A registers.  The block's x is converted once
// into shared memory in the exact lane order of the B fragments.
//
// Column order inside an mma.  The reduction order of a dot product is free,
// so the 16 k slots of each mma are bound to columns to suit the loads: lane
// (g = lane/4, t = lane%4) loads 16 bytes of row g and of row g+8 at column
// 64*kb + 16*t, and mma i (0..3) of K-block kb binds its slots 2t, 2t+1,
// 2t+8, 2t+9 to columns 64*kb + 16*t + 4*i + 0, 1, 2, 3 -- in A and in B alike.
//
// Scales.  After the four mma of a 64-column block the lane holds, for rows
// g and g+8 and vector 4j+t, (sum w * hi, sum w * lo); it adds them, undoes
// 2^E and multiplies by the row's E8M0 scale of that block (one float32
// multiply and FMA per row and vector).  So every 64-column block must lie in
// one scale column block; rows may change scale row anywhere.
//
// Work split.  A block owns tiles of 16 rows, in grid-stride order; its warps
// split the row's 64-column blocks and walk them in steps of four, loading
// the next step (or the next tile's first) before computing the current one.
// At the end of a tile each warp writes its partial sums to shared memory
// (double buffered, one barrier per tile) and 16 * batch threads add the
// warps' partials in a fixed order, so results are deterministic.
//
// Fix-up.  A result that is not finite is recomputed by the exact
// per-element path (saturating decode), which gives 0x7F / 0xFF codes (NaN
// under the hardware conversion), NaN scales and non-finite x their
// per-element meaning; blocks of x holding Inf or NaN are flagged so that
// their rows always take that path.
// ---------------------------------------------------------------------------

constexpr int kMmaKS = 4;  // 64-column blocks per warp step

// One warp step: rows r0+g and r0+g+8, K-blocks kb0 .. kb0+3, and the E8M0
// codes of the two rows for those blocks.
struct MmaStep {
    uint4 w[2][kMmaKS];
    unsigned s[2][kMmaKS];
};

// Rows past R re-read row R-1 and K-blocks past the warp's range re-read its
// last one (in bounds, results unused), so no load is predicated.
__device__ __forceinline__ void mma_load(MmaStep &st, const F8Args &a, const int *cb64, int64_t ra, int64_t rb,
                                         int64_t sra, int64_t srb, int kb0, int kb_hi, int t) {
    const uint8_t *pa = a.w + ra * a.C + 16 * t, *pb = a.w + rb * a.C + 16 * t;
#pragma unroll
    for (int k = 0; k < kMmaKS; k++) {
        const int kb = min(kb0 + k, kb_hi - 1);
        st.w[0][k] = ld_stream(pa + int64_t(kb) * 64);
        st.w[1][k] = ld_stream(pb + int64_t(kb) * 64);
        const int cb = cb64[kb];
        st.s[0][k] = __ldg(a.scale + sra + cb);
        st.s[1][k] = __ldg(a.scale + srb + cb);
    }
}

// Four E4M3 bytes -> two f16 pairs (bytes 0-1 -> lo, bytes 2-3 -> hi).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(static_cast<unsigned short>(two_bytes)));
    return out;
}

// tot[j][h] += sum over the step's K-blocks of row (g + 8h), vector 4j+t.
// frag is [K-step][lane][NJ] of (b0b1, b2b3); fv is [K-block][4*NJ] of 2^-E.
template <int NJ>
__device__ __forceinline__ void mma_compute(float (&tot)[NJ][2], const MmaStep &st, const uint2 *frag,
                                            const float *fv, int kb0, int kb_hi, int lane) {
    const int t = lane & 3;
#pragma unroll
    for (int k = 0; k < kMmaKS; k++) {
        const int kb = kb0 + k;
        if (kb >= kb_hi) break;  // warp-uniform
        float acc[NJ][4];
#pragma unroll
        for (int j = 0; j < NJ; j++) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t wa = word_of(st.w[0][k], i), wb = word_of(st.w[1][k], i);
            const uint32_t a0 = e4m3x2_to_f16x2(wa & 0xffffu), a1 = e4m3x2_to_f16x2(wb & 0xffffu);
            const uint32_t a2 = e4m3x2_to_f16x2(wa >> 16), a3 = e4m3x2_to_f16x2(wb >> 16);
            const uint2 *fr = frag + (int64_t(kb * 4 + i) * 32 + lane) * NJ;
            if constexpr (NJ == 2) {
                const uint4 b = *reinterpret_cast<const uint4 *>(fr);
                mma_16816(acc[0], a0, a1, a2, a3, b.x, b.y);
                mma_16816(acc[1], a0, a1, a2, a3, b.z, b.w);
            } else {
                const uint2 b = fr[0];
                mma_16816(acc[0], a0, a1, a2, a3, b.x, b.y);
            }
        }
        const float sa = e8m0_value(st.s[0][k]), sb = e8m0_value(st.s[1][k]);
#pragma unroll
        for (int j = 0; j < NJ; j++) {
            const float f = fv[kb * 4 * NJ + 4 * j + t];
            tot[j][0] = fmaf((acc[j][0] + acc[j][1]) * f, sa, tot[j][0]);
            tot[j][1] = fmaf((acc[j][2] + acc[j][3]) * f, sb, tot[j][1]);
        }
    }
}

// x -> B fragments in shared memory: one warp per (64-column block kb,
// vector slot v); lane l holds columns 64*kb + 2l and 2l+1.
template <int NJ>
__device__ __forceinline__ void mma_prepare_x(const F8Args &a, int batch, int nkb, uint2 *frag, float *fv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    uint32_t *fw = reinterpret_cast<uint32_t *>(frag);
    for (int job = warp; job < nkb * 4 * NJ; job += nw) {
        const int kb = job / (4 * NJ), v = job - kb * (4 * NJ);
        float2 xv = make_float2(0.0f, 0.0f);
        if (v < batch) xv = __ldg(reinterpret_cast<const float2 *>(a.x + int64_t(v) * a.C + int64_t(kb) * 64) + lane);
        uint32_t hi, lo;
        float f;
        split_block(xv, hi, lo, f);
        if (lane == 0) fv[kb * 4 * NJ + v] = f;
        // destination: K-step 4*kb + i, lanes (g' = 2*(v%4) + {0: hi, 1: lo}, t'), half e
        const int tp = lane >> 3, i = (lane & 7) >> 1, e = lane & 1;
        const int j = v >> 2, gh = 2 * (v & 3);
        const int64_t step = int64_t(kb * 4 + i) * 32;
        fw[((step + gh * 4 + tp) * NJ + j) * 2 + e] = hi;
        fw[((step + (gh + 1) * 4 + tp) * NJ + j) * 2 + e] = lo;
    }
}

// Shared memory of the mma kernel for C columns (C % 64 == 0) and NW warps.
__host__ __device__ inline size_t mma_smem_bytes(int64_t C, int NJ, int NW) {
    const int64_t nkb = C / 64;
    return size_t(nkb * 4 * 32 * NJ * 8      // B fragments
                  + nkb * 4 * NJ * 4          // 2^-E per (K-block, vector slot)
                  + 2 * NW * NJ * 32 * 8      // partial sums, double buffered
                  + nkb * 4);                 // scale column of each K-block
}

// The exact per-element evaluation of one output, as the tile epilogue's
// fix-up of non-finite results (warp-collective).
struct F8Exact {
    const F8Args &a;
    __device__ __forceinline__ float operator()(int64_t r, int v) const { return f8_row_exact(a, r, v, nullptr); }
};

// Argmax epilogue of the mma kernels: the 16 reducer threads of vector v
// (lanes 16*(v%2) .. +15 of one warp) reduce their bests, and the block's
// best for every vector goes to ws[blockIdx.x * batch + v].
__device__ __forceinline__ void mma_argmax_store(float best_v, int64_t best_i, const F8Args &a, int batch) {
    const int warp = threadIdx.x >> 5, o = threadIdx.x;
    if (warp >= (16 * batch + 31) / 32) return;
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) {
        const float ov = __shfl_xor_sync(kFull, best_v, d);
        const int64_t oi = __shfl_xor_sync(kFull, best_i, d);
        if (arg_better(ov, oi, best_v, best_i)) {
            best_v = ov;
            best_i = oi;
        }
    }
    if (o < 16 * batch && (o & 15) == 0) {
        ArgBest r;
        r.v = best_v;
        r.pad = 0;
        r.i = best_i;
        a.ws[int64_t(blockIdx.x) * batch + (o >> 4)] = r;
    }
}

template <int NJ, bool AM>
__global__ void __launch_bounds__(512, 1) f8_mma_kernel(F8Args a, int batch) {
    extern __shared__ __align__(16) unsigned char mma_smem[];
    const int nkb = int(a.C >> 6);
    const int NW = blockDim.x >> 5;
    uint2 *frag = reinterpret_cast<uint2 *>(mma_smem);
    float *fv = reinterpret_cast<float *>(mma_smem + size_t(nkb) * 4 * 32 * NJ * 8);
    float *red = fv + nkb * 4 * NJ;  // [2][NW][NJ][32] x (row g, row g+8)
    int *cb64 = reinterpret_cast<int *>(red + 2 * NW * NJ * 32 * 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2;
    for (int kb = threadIdx.x; kb < nkb; kb += blockDim.x) cb64[kb] = int((int64_t(kb) * 64 * a.SC) / a.C);
    pdl_wait();
    pdl_trigger();
    __syncthreads();

    const int kb_lo = warp * nkb / NW, kb_hi = (warp + 1) * nkb / NW;
    const int nsteps = (kb_hi - kb_lo + kMmaKS - 1) / kMmaKS;
    const int64_t ntiles = (a.R + 15) >> 4;
    float best_v = -INFINITY;
    int64_t best_i = INT64_MAX;

    int64_t tile = blockIdx.x;
    if (tile < ntiles) {  // block-uniform (no early return: the argmax epilogue has a barrier)
        auto rows_of = [&](int64_t tl, int64_t &ra, int64_t &rb, int64_t &sra, int64_t &srb) {
            ra = min(tl * 16 + g, a.R - 1);
            rb = min(tl * 16 + g + 8, a.R - 1);
            sra = (ra * a.SR / a.R) * a.SC;
            srb = (rb * a.SR / a.R) * a.SC;
        };
        int64_t ra, rb, sra, srb;
        rows_of(tile, ra, rb, sra, srb);
        int step = 0;
        MmaStep cur;
        mma_load(cur, a, cb64, ra, rb, sra, srb, kb_lo, kb_hi, lane & 3);
        mma_prepare_x<NJ>(a, batch, nkb, frag, fv);  // overlaps the first loads
        __syncthreads();

        float tot[NJ][2];
#pragma unroll
        for (int j = 0; j < NJ; j++) tot[j][0] = tot[j][1] = 0.0f;
        int buf = 0;
        while (true) {
            int stepn = step + 1;
            int64_t tilen = tile;
            if (stepn == nsteps) {
                stepn = 0;
                tilen = tile + gridDim.x;
            }
            const bool has_next = tilen < ntiles;
            int64_t ran = ra, rbn = rb, sran = sra, srbn = srb;
            MmaStep nxt;
            if (has_next) {
                if (tilen != tile) rows_of(tilen, ran, rbn, sran, srbn);
                mma_load(nxt, a, cb64, ran, rbn, sran, srbn, kb_lo + kMmaKS * stepn, kb_hi, lane & 3);
            }
            mma_compute<NJ>(tot, cur, frag, fv, kb_lo + kMmaKS * step, kb_hi, lane);

            if (step == nsteps - 1) {
                mma::tile_epilogue<NJ, AM>(tot, red, buf, NW, batch, a.R, a.y, tile * 16, best_v, best_i, F8Exact{a}, arg_better);
                buf ^= 1;
            }
            if (!has_next) break;
            cur = nxt;
            step = stepn;
            tile = tilen;
            ra = ran;
            rb = rbn;
            sra = sran;
            srb = srbn;
        }
    }
    if (AM) mma_argmax_store(best_v, best_i, a, batch);
}

// ---------------------------------------------------------------------------
// Staged tensor-core kernel (C <= 4096, every warp <= four 64-column blocks).
//
// The kernel above keeps one 4 KB step per warp in flight in registers, which
// is ~64 KB per SM: at the loaded DRAM latency that caps it near 4.5-5 TB/s.
// Here the weights go through a three-deep ring of cp.async copies
// (global -> shared, 16 bytes per lane, no registers held), so two tiles per
// warp (~128 KB per SM) are always in flight; cp.async.wait_group is the only
// wait.  Each warp owns the same <= 4 column blocks of every tile of its
// block, so its B fragments and 2^-E factors live in registers, built once.
// Arithmetic, epilogue and fix-up are those of the kernel above (the split
// of the row among warps can differ, and with it the order of the partial
// sums).
//
// Ring layout: warp w, stage s, row rho (16), 16-byte chunk position; the
// copies are coalesced whole lines and the reads follow the fragment order,
// so a __syncwarp after cp.async.wait_group publishes the lanes' copies.
// ---------------------------------------------------------------------------

// Scale-row offset (row * SR / R) * SC of row r; `div32` when R * SR < 2^32.
__device__ __forceinline__ int64_t scale_row_offset(const F8Args &a, int64_t r, bool div32) {
    const int64_t q = div32 ? int64_t(uint32_t(uint64_t(r) * uint64_t(a.SR)) / uint32_t(a.R)) : r * a.SR / a.R;
    return q * a.SC;
}

template <int NJ, int NK, bool AM>
__global__ void __launch_bounds__(512, 1) f8_mma_staged_kernel(F8Args a, int batch, int div32) {
    extern __shared__ __align__(16) unsigned char st_smem[];
    constexpr int NCH = 4 * NK;                 // 16-byte chunks per row and warp
    constexpr int SLOT = 16 * NCH * 16;         // bytes per warp and stage
    const int NW = blockDim.x >> 5;             // warp w owns K-blocks [w NK, w NK + NK)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int kb_lo = warp * NK;
    const uint32_t ring = uint32_t(__cvta_generic_to_shared(st_smem)) + uint32_t(warp * kRing * SLOT);
    const uint4 *ring_g = reinterpret_cast<const uint4 *>(st_smem + size_t(warp) * kRing * SLOT);
    float *red = reinterpret_cast<float *>(st_smem + size_t(NW) * kRing * SLOT);

    // scale column of every K-block (depends only on shapes)
    int *cb64 = reinterpret_cast<int *>(red + 2 * NW * NJ * 32 * 2);
    for (int kb = threadIdx.x; kb < NW * NK; kb += blockDim.x) cb64[kb] = int((int64_t(kb) * 64 * a.SC) / a.C);

    pdl_wait();
    pdl_trigger();
    __syncthreads();

    const int64_t ntiles = (a.R + 15) >> 4;
    const int64_t gstride = gridDim.x;
    float best_v = -INFINITY;
    int64_t best_i = INT64_MAX;
    // E8M0 codes of rows g and g+8 for this warp's K-blocks of tile tl (lane l
    // computes the scale row of row l % 16)
    auto load_scales = [&](int64_t tl, unsigned (&sa)[NK], unsigned (&sb)[NK]) {
        const int64_t my_off = scale_row_offset(a, min(tl * 16 + (lane & 15), a.R - 1), div32 != 0);
        const int64_t off_a = __shfl_sync(kFull, my_off, g), off_b = __shfl_sync(kFull, my_off, g + 8);
#pragma unroll
        for (int k = 0; k < NK; k++) {
            const int cb = cb64[kb_lo + k];
            sa[k] = __ldg(a.scale + off_a + cb);
            sb[k] = __ldg(a.scale + off_b + cb);
        }
    };
    if (int64_t(blockIdx.x) < ntiles) {  // block-uniform
        // the first kRing - 1 tiles go out before the B fragments are built
#pragma unroll
        for (int st = 0; st < kRing - 1; st++) {
            const int64_t tl = blockIdx.x + st * gstride;
            if (tl < ntiles) mma::issue_tile<NK>(ring + uint32_t(st * SLOT), a.w, a.R, a.C, tl, kb_lo, lane);
            cp_async_commit();
        }
        unsigned sa[NK], sb[NK];
        load_scales(blockIdx.x, sa, sb);
        mma::StagedB<NJ> B;
        mma::build_b<NJ>(B, a.x, a.C, batch, kb_lo, NK, lane);

        float tot[NJ][2];
#pragma unroll
        for (int j = 0; j < NJ; j++) tot[j][0] = tot[j][1] = 0.0f;
        int buf = 0, slot = 0;
        for (int64_t tl = blockIdx.x; tl < ntiles; tl += gstride) {
            // next copies: tile tl + (kRing-1) strides into the slot freed last
            // round (every lane's reads of it ended before the last barrier)
            {
                const int64_t tn = tl + (kRing - 1) * gstride;
                int sn = slot + kRing - 1;
                if (sn >= kRing) sn -= kRing;
                if (tn < ntiles) mma::issue_tile<NK>(ring + uint32_t(sn * SLOT), a.w, a.R, a.C, tn, kb_lo, lane);
                cp_async_commit();
            }
            // next tile's scale codes, one tile ahead
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
                const uint4 wa4 = mma::row_chunk<NK>(src, g, 4 * k + t);
                const uint4 wb4 = mma::row_chunk<NK>(src, g + 8, 4 * k + t);
                // NJ == 1: two accumulator chains (even / odd mma) for latency
                constexpr int NA = NJ == 1 ? 2 : 1;
                float acc[NA][NJ][4];
#pragma unroll
                for (int q = 0; q < NA; q++)
#pragma unroll
                    for (int j = 0; j < NJ; j++) acc[q][j][0] = acc[q][j][1] = acc[q][j][2] = acc[q][j][3] = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    uint32_t a0, a2, a1, a3;
                    e4m3x4_to_f16x2x2(word_of(wa4, i), a0, a2);
                    e4m3x4_to_f16x2x2(word_of(wb4, i), a1, a3);
#pragma unroll
                    for (int j = 0; j < NJ; j++)
                        mma_16816(acc[i % NA][j], a0, a1, a2, a3, B.b[k][i][j][0], B.b[k][i][j][1]);
                }
                const float s_a = e8m0_value(sa[k]), s_b = e8m0_value(sb[k]);
#pragma unroll
                for (int j = 0; j < NJ; j++) {
                    const float f = B.f[k][j];
                    float ha = acc[0][j][0] + acc[0][j][1], hb = acc[0][j][2] + acc[0][j][3];
                    if (NA == 2) {
                        ha += acc[NA - 1][j][0] + acc[NA - 1][j][1];
                        hb += acc[NA - 1][j][2] + acc[NA - 1][j][3];
                    }
                    tot[j][0] = fmaf(ha * f, s_a, tot[j][0]);
                    tot[j][1] = fmaf(hb * f, s_b, tot[j][1]);
                }
            }
            mma::tile_epilogue<NJ, AM>(tot, red, buf, NW, batch, a.R, a.y, tl * 16, best_v, best_i, F8Exact{a}, arg_better);
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
    if (AM) mma_argmax_store(best_v, best_i, a, batch);
}

// Final pass of the argmax: one block reduces the [nblocks, B] partials.
__global__ void __launch_bounds__(256) argmax_reduce_kernel(const ArgBest *ws, int nblocks, int B,
                                                            int64_t *out_index, float *out_value) {
    pdl_wait();
    pdl_trigger();
    __shared__ float sv[256];
    __shared__ int64_t si[256];
    for (int k = 0; k < B; k++) {
        float bv = -INFINITY;
        int64_t bi = INT64_MAX;
        for (int b = threadIdx.x; b < nblocks; b += blockDim.x) {
            const ArgBest e = ws[int64_t(b) * B + k];
            if (arg_better(e.v, e.i, bv, bi)) {
                bv = e.v;
                bi = e.i;
            }
        }
        sv[threadIdx.x] = bv;
        si[threadIdx.x] = bi;
        __syncthreads();
        for (int st = blockDim.x / 2; st > 0; st >>= 1) {
            if (threadIdx.x < st && arg_better(sv[threadIdx.x + st], si[threadIdx.x + st], sv[threadIdx.x],
                                               si[threadIdx.x])) {
                sv[threadIdx.x] = sv[threadIdx.x + st];
                si[threadIdx.x] = si[threadIdx.x + st];
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            out_index[k] = si[0];
            out_value[k] = sv[0];
        }
        __syncthreads();
    }
}

// True when every `width`-column chunk maps to a single scale block: the
// first column of each block b, ceil(b*C/SC), is a multiple of `width`.
bool chunks_uniform(int64_t C, int64_t SC, int64_t width = 16) {
    for (int64_t b = 1; b < SC; b++) {
        const int64_t start = (b * C + SC - 1) / SC;
        if (start % width != 0) return false;
    }
    return true;
}

// The tensor-core kernel: C % 64 == 0 with at least four 64-column blocks
// (one warp per block, and the tile epilogue needs 16 * batch <= 128 threads),
// 16-byte aligned w and x, every 64-column block inside one scale block, and
// its shared memory in reach.
constexpr size_t kMmaSmemMax = 200 * 1024;
bool mma_fits(const F8Args &a, int batch) {
    if (batch < 2 || a.C % 64 != 0 || a.C < 256) return false;
    if (reinterpret_cast<uintptr_t>(a.w) % 16 != 0 || reinterpret_cast<uintptr_t>(a.x) % 16 != 0) return false;
    const int NJ = (batch + 3) / 4;
    const int NW = a.C / 64 < 16 ? int(a.C / 64) : 16;
    if (mma_smem_bytes(a.C, NJ, NW) > kMmaSmemMax) return false;
    return chunks_uniform(a.C, a.SC, 64);
}

template <int NJ, int NK, bool AM>
qmv_status launch_mma_staged(const F8Args &a, int batch, cudaStream_t s, int &blocks_out) {
    const int NW = int(a.C / 64 / NK);
    const size_t smem = mma::staged_smem_bytes(NW, NK, NJ, size_t(NW) * NK * 4);  // + scale columns
    auto kern = f8_mma_staged_kernel<NJ, NK, AM>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int64_t ntiles = (a.R + 15) / 16;
    int64_t blocks = int64_t(occupancy(kp, 32 * NW, smem)) * sm_count();
    if (blocks > ntiles) blocks = ntiles;
    if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
    blocks_out = int(blocks);
    // R * SR < 2^32: the scale-row index takes a 32-bit division
    const int div32 = (a.R < (int64_t(1) << 32) && a.SR <= (int64_t(0xffffffff) / a.R)) ? 1 : 0;
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(32 * NW), smem, s, a, batch, div32));
}

template <int NJ, bool AM>
qmv_status launch_mma(const F8Args &a, int batch, cudaStream_t s, int &blocks_out) {
    switch (mma::staged_nk(a.C, batch)) {
        case 4: return launch_mma_staged<NJ, 4, AM>(a, batch, s, blocks_out);
        case 2: return launch_mma_staged<NJ, 2, AM>(a, batch, s, blocks_out);
        case 1: return launch_mma_staged<NJ, 1, AM>(a, batch, s, blocks_out);
        default: break;
    }
    const int NW = a.C / 64 < 16 ? int(a.C / 64) : 16;
    const size_t smem = mma_smem_bytes(a.C, NJ, NW);
    auto kern = f8_mma_kernel<NJ, AM>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int64_t ntiles = (a.R + 15) / 16;
    int64_t blocks = int64_t(occupancy(kp, 32 * NW, smem)) * sm_count();
    if (blocks > ntiles) blocks = ntiles;
    if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
    blocks_out = int(blocks);
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(32 * NW), smem, s, a, batch));
}

template <int B, bool AM, int T = (B <= 2) ? 8 : 4, bool PF = false, bool GS = true>
qmv_status launch_fast(const F8Args &a, cudaStream_t s, int &blocks_out) {
    const size_t smem = size_t(a.C >> 4) * sizeof(int);
    auto kern = f8_fast_kernel<B, T, PF, GS, AM>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int64_t capacity = int64_t(occupancy(kp, 256, smem)) * sm_count() * 8;  // resident warps
    int blocks;
    cudaError_t e;
    if ((a.R + T - 1) / T < 4 * capacity) {
        // too few tiles to keep a full grid streaming: load whole rows at once
        constexpr int TS = 2, NSTEP = (B <= 2) ? 8 : 4;
        auto rk = f8_rows_kernel<B, TS, NSTEP, AM>;
        const void *rp = reinterpret_cast<const void *>(rk);
        if (!allow_smem(rp, smem)) return QMV_ERR_CUDA;
        blocks = grid_blocks(rp, 256, smem, (a.R + TS - 1) / TS);
        if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
        e = launch_pdl(rk, dim3(unsigned(blocks)), dim3(256), smem, s, a);
    } else {
        blocks = grid_blocks(kp, 256, smem, (a.R + T - 1) / T);
        if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
        e = launch_pdl(kern, dim3(unsigned(blocks)), dim3(256), smem, s, a);
    }
    blocks_out = blocks;
    return from_cuda(e);
}

template <int B, bool AM>
qmv_status launch_general(const F8Args &a, cudaStream_t s, int &blocks_out) {
    const void *kp = reinterpret_cast<const void *>(f8_general_kernel<B, AM>);
    int blocks = grid_blocks(kp, 256, 0, a.R);
    if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
    blocks_out = blocks;
    return from_cuda(launch_pdl(f8_general_kernel<B, AM>, dim3(unsigned(blocks)), dim3(256), 0, s, a));
}

template <bool AM>
qmv_status launch_any(const F8Args &a, int batch, cudaStream_t s, int &blocks) {
    const bool fast = (a.C % 16 == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(a.x) % 16 == 0) && (a.C / 16) * 4 <= 200 * 1024 &&
                      chunks_uniform(a.C, a.SC);
    if (a.R > 0 && mma_fits(a, batch))
        return batch <= 4 ? launch_mma<1, AM>(a, batch, s, blocks) : launch_mma<2, AM>(a, batch, s, blocks);
    if (fast) {
        switch (batch) {
            case 1: return launch_fast<1, AM>(a, s, blocks);
            case 2: return launch_fast<2, AM>(a, s, blocks);
            case 3: return launch_fast<3, AM>(a, s, blocks);
            case 4: return launch_fast<4, AM>(a, s, blocks);
            case 5: return launch_fast<5, AM>(a, s, blocks);
            case 6: return launch_fast<6, AM>(a, s, blocks);
            case 7: return launch_fast<7, AM>(a, s, blocks);
            default: return launch_fast<8, AM>(a, s, blocks);
        }
    }
    switch (batch) {
        case 1: return launch_general<1, AM>(a, s, blocks);
        case 2: return launch_general<2, AM>(a, s, blocks);
        case 3: return launch_general<3, AM>(a, s, blocks);
        case 4: return launch_general<4, AM>(a, s, blocks);
        case 5: return launch_general<5, AM>(a, s, blocks);
        case 6: return launch_general<6, AM>(a, s, blocks);
        case 7: return launch_general<7, AM>(a, s, blocks);
        default: return launch_general<8, AM>(a, s, blocks);
    }
}

}  // namespace

qmv_status launch_f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                            int64_t SC, const float *x, int batch, float *y, cudaStream_t s) {
    F8Args a{w, scale, x, y, R, C, SR, SC, nullptr};
    int blocks = 0;
    return launch_any<false>(a, batch, s, blocks);
}

qmv_status launch_f8_matvec_argmax(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                                   int64_t SC, const float *x, int batch, float *y, int64_t *out_index,
                                   float *out_value, void *workspace, cudaStream_t s) {
    F8Args a{w, scale, x, y, R, C, SR, SC, reinterpret_cast<ArgBest *>(workspace)};
    int blocks = 0;
    qmv_status st = launch_any<true>(a, batch, s, blocks);
    if (st != QMV_OK) return st;
    return from_cuda(launch_pdl(argmax_reduce_kernel, dim3(1), dim3(256), 0, s,
                                static_cast<const ArgBest *>(a.ws), blocks, batch, out_index, out_value));
}

}  // namespace qmv
