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
#include "f8_common.cuh"

namespace qmv {
namespace f8 {
namespace {

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
    if (AM) {
        __shared__ __align__(16) unsigned char arg_scratch[sizeof(ArgScratch)];
        block_best_store<B>(best, a.ws);
        argmax_complete(a, B, arg_scratch);
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
    const float s0 = dev::e8m0(__ldg(srow0 + cb));
    auto scale_of = [&](int t) -> float {
        return UNIFORM ? s0 : dev::e8m0(__ldg(srow0 + int64_t((dpack >> (4 * t)) & 15u) * a.SC + cb));
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

// A warp's running argmax best kept in shared memory [warp][B] by lane 0
// (blocks of at most 8 warps; the values offered are warp-uniform), so it
// takes no registers from the streaming accumulators.  store_block reduces
// the block's warps in warp order into ws[blockIdx.x * B + k]; every thread
// of the block calls it.
template <int B>
struct SmemBest {
    static __device__ __forceinline__ float (&vals())[8][B] {
        __shared__ float v[8][B];
        return v;
    }
    static __device__ __forceinline__ int64_t (&rows())[8][B] {
        __shared__ int64_t r[8][B];
        return r;
    }
    __device__ __forceinline__ void init() {
        if ((threadIdx.x & 31) == 0) {
#pragma unroll
            for (int k = 0; k < B; k++) {
                vals()[threadIdx.x >> 5][k] = -INFINITY;
                rows()[threadIdx.x >> 5][k] = INT64_MAX;
            }
        }
    }
    __device__ __forceinline__ void offer(int k, float val, int64_t row) {
        const int w = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0 && arg_better(val, row, vals()[w][k], rows()[w][k])) {
            vals()[w][k] = val;
            rows()[w][k] = row;
        }
    }
    __device__ __forceinline__ void store_block(ArgBest *ws) {
        __syncthreads();
        if (threadIdx.x < B) {
            const int k = threadIdx.x, nw = blockDim.x >> 5;
            float bv = vals()[0][k];
            int64_t bi = rows()[0][k];
            for (int w2 = 1; w2 < nw; w2++)
                if (arg_better(vals()[w2][k], rows()[w2][k], bv, bi)) {
                    bv = vals()[w2][k];
                    bi = rows()[w2][k];
                }
            ArgBest r;
            r.v = bv;
            r.pad = 0;
            r.i = bi;
            ws[int64_t(blockIdx.x) * B + k] = r;
        }
    }
};

// Tile epilogue: reduce each row's sums across the warp (fixed order), fall
// back to the exact per-element evaluation for rows that came out NaN, store.
// With AM, the tile's best row per vector is found in registers first (the
// values are warp-uniform, so every lane agrees), and offered once.
template <int B, int T, bool AM, typename Best>
__device__ __forceinline__ void finish_tile(typename AccOf<B>::type (&acc)[T][B], const F8Args &a, int64_t r0,
                                            int rows, int lane, Best &best) {
    float tv[B];
    int ti[B];
#pragma unroll
    for (int v = 0; v < B; v++) {
        tv[v] = -INFINITY;
        ti[v] = T;
    }
#pragma unroll
    for (int t = 0; t < T; t++) {
#pragma unroll
        for (int v = 0; v < B; v++) {
            float val = warp_sum(acc_total(acc[t][v]));
            acc_zero(acc[t][v]);
            if (t < rows) {
                if (isnan(val)) val = f8_row_exact(a, r0 + t, v, nullptr);
                if (AM && arg_better(val, t, tv[v], ti[v])) {
                    tv[v] = val;
                    ti[v] = t;
                }
                if (lane == 0 && (!AM || a.y)) a.y[int64_t(v) * a.R + r0 + t] = val;
            }
        }
    }
    if (AM) {
#pragma unroll
        for (int v = 0; v < B; v++)
            if (ti[v] < T) best.offer(v, tv[v], r0 + ti[v]);
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
    pdl_trigger();
    const int64_t nchunk = a.C >> 4;
    // (depends only on the shapes: runs before the wait)
    for (int64_t ch = threadIdx.x; ch < nchunk; ch += blockDim.x)
        chunk_cb[ch] = int((ch * 16 * a.SC) / a.C);

    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    // GS: tiles in grid-stride order (all warps sweep one region of the
    // matrix together); otherwise each warp owns an even contiguous share.
    const int64_t row_end = GS ? a.R : a.R * (wid + 1) / nwarps;
    int64_t r0 = GS ? wid * T : a.R * wid / nwarps;
    const int64_t tile_stride = GS ? nwarps * T : T;
    // the first step of the first tile goes out before the dependency wait
    // (the weights never depend on the preceding kernel); the argmax variant,
    // tighter on registers, loads it after the wait
    uint4 cur[T];
    if (!AM && r0 < row_end) load_step<T>(cur, a, r0, int(min(int64_t(T), row_end - r0)), lane, nchunk);
    pdl_wait();
    __syncthreads();
    // the argmax's running best of each warp lives in shared memory (lane 0
    // keeps it; the values it is offered are warp-uniform), which leaves the
    // registers to the streaming accumulators; each tile offers only its best
    SmemBest<B> best;
    best.init();
    if (r0 < row_end) {  // (no early return: the argmax epilogue has a barrier)
    const int iters = int((nchunk + 31) >> 5);

    int rows = int(min(int64_t(T), row_end - r0));
    int j = 0;
    if (AM) load_step<T>(cur, a, r0, rows, lane, nchunk);

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
    if (AM) {
        __shared__ __align__(16) unsigned char arg_scratch[sizeof(ArgScratch)];
        best.store_block(a.ws);
        argmax_complete(a, B, arg_scratch);
    }
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
    pdl_trigger();
    const int64_t nchunk = a.C >> 4;
    for (int64_t ch = threadIdx.x; ch < nchunk; ch += blockDim.x)
        chunk_cb[ch] = int((ch * 16 * a.SC) / a.C);
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t ntiles = (a.R + T - 1) / T;
    const int64_t tile0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    // the first steps of this warp's first tile go out before the wait (the
    // weights never depend on the preceding kernel)
    uint4 d[NSTEP][T];
    if (tile0 < ntiles) {
        const int rows0 = int(min(int64_t(T), a.R - tile0 * T));
#pragma unroll
        for (int st = 0; st < NSTEP; st++) load_step<T>(d[st], a, tile0 * T, rows0, lane + 32 * st, nchunk);
    }
    pdl_wait();
    __syncthreads();

    typename AccOf<B>::type acc[T][B];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int v = 0; v < B; v++) acc_zero(acc[t][v]);

    WarpBest<B> best;
    best.init();
    for (int64_t tile = tile0; tile < ntiles; tile += nwarps) {
        const int64_t r0 = tile * T;
        const int rows = int(min(int64_t(T), a.R - r0));
        const uint8_t *srow0;
        uint32_t dpack;
        const bool uniform = setup_scale<T>(a, r0, rows, srow0, dpack);
        for (int64_t base = 0; base < nchunk; base += 32 * NSTEP) {
            if (tile != tile0 || base != 0) {
#pragma unroll
                for (int st = 0; st < NSTEP; st++) load_step<T>(d[st], a, r0, rows, base + lane + 32 * st, nchunk);
            }
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
    if (AM) {
        __shared__ __align__(16) unsigned char arg_scratch[sizeof(ArgScratch)];
        block_best_store<B>(best, a.ws);
        argmax_complete(a, B, arg_scratch);
    }
}

// ---------------------------------------------------------------------------
// Split-row kernel (batch 1, C from 4096 to 16384 columns, few rows): a block
// of 8 warps takes a tile of T rows and every warp a share of its columns --
// lane l of warp w reads the chunks l + 32 (w + 8 s), s < NS, of each row --
// so the block requests the tile's T * C bytes with all 256 threads at once,
// and a matrix of up to (resident blocks) x T rows goes out in one wave of
// loads, issued before the dependency wait.  The warps' row sums meet in
// shared memory and are added in warp order; warp t finishes row t (NaN
// fix-up, store, argmax offer).  NS * T = 8 chunks in flight per thread.
// ---------------------------------------------------------------------------
constexpr int kSplitWarps = 8;

template <int T, int NS, bool AM>
__global__ void __launch_bounds__(256, 4) f8_split_kernel(F8Args a) {
    static_assert(T <= kSplitWarps, "warp t finishes row t");
    extern __shared__ int chunk_cb[];
    __shared__ float part[kSplitWarps][T];
    pdl_trigger();
    const int64_t nchunk = a.C >> 4;
    for (int64_t ch = threadIdx.x; ch < nchunk; ch += blockDim.x)
        chunk_cb[ch] = int((ch * 16 * a.SC) / a.C);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // one tile per block (the launcher makes the grid cover every tile)
    const int64_t r0 = int64_t(blockIdx.x) * T;
    const int rows = int(min(int64_t(T), a.R - r0));
    uint4 d[NS][T];
#pragma unroll
    for (int st = 0; st < NS; st++)  // weights only: before the wait
        load_step<T>(d[st], a, r0, rows, lane + 32 * (warp + kSplitWarps * st), nchunk);
    pdl_wait();
    __syncthreads();

    const uint8_t *srow0;
    uint32_t dpack;
    const bool uniform = setup_scale<T>(a, r0, rows, srow0, dpack);
    float acc[T][1];
#pragma unroll
    for (int t = 0; t < T; t++) acc[t][0] = 0.0f;
#pragma unroll
    for (int st = 0; st < NS; st++) {
        const int64_t ch = lane + 32 * (warp + kSplitWarps * st);
        if (ch < nchunk) {
            if (uniform)
                compute_step<1, T, true>(acc, d[st], a, srow0, dpack, chunk_cb[ch], ch);
            else
                compute_step<1, T, false>(acc, d[st], a, srow0, dpack, chunk_cb[ch], ch);
        }
    }
#pragma unroll
    for (int t = 0; t < T; t++) {
        const float pv = warp_sum(acc[t][0]);
        if (lane == 0) part[warp][t] = pv;
    }
    __syncthreads();
    WarpBest<1> best;
    best.init();
    if (warp < rows) {  // warp-uniform
        float val = part[0][warp];
#pragma unroll
        for (int w2 = 1; w2 < kSplitWarps; w2++) val += part[w2][warp];
        if (isnan(val)) val = f8_row_exact(a, r0 + warp, 0, nullptr);
        if (AM) best.offer(0, val, r0 + warp);
        if (lane == 0 && (!AM || a.y)) a.y[r0 + warp] = val;
    }
    if (AM) {
        __shared__ __align__(16) unsigned char arg_scratch[sizeof(ArgScratch)];
        block_best_store<1>(best, a.ws);
        argmax_complete(a, 1, arg_scratch);
    }
}

// Steps per thread of the split kernel for C columns: 1, 2 or 4 (0: not taken).
inline int split_steps(int64_t C) {
    const int64_t nchunk = C >> 4;
    if (nchunk < 32 * kSplitWarps) return 0;
    for (int ns = 1; ns <= 4; ns *= 2)
        if (nchunk <= int64_t(32) * kSplitWarps * ns) return ns;
    return 0;
}

template <int T, int NS, bool AM>
int split_capacity(size_t smem) {
    const void *kp = reinterpret_cast<const void *>(f8_split_kernel<T, NS, AM>);
    if (!allow_smem(kp, smem)) return 0;
    return occupancy(kp, 256, smem) * sm_count();
}

// Whether the split kernel takes this batch-1 call (the fast kernel's
// requirements hold): C in [4096, 16384] and every tile resident at once.
template <bool AM>
bool split_fits(const F8Args &a) {
    const int ns = split_steps(a.C);
    if (ns == 0) return false;
    const size_t smem = size_t(a.C >> 4) * sizeof(int);
    const int T = 8 / ns;
    const int cap = ns == 1 ? split_capacity<8, 1, AM>(smem)
                  : ns == 2 ? split_capacity<4, 2, AM>(smem)
                            : split_capacity<2, 4, AM>(smem);
    return (a.R + T - 1) / T <= int64_t(cap);
}

template <int T, int NS, bool AM>
qmv_status launch_split_t(const F8Args &a, cudaStream_t s, int &blocks_out) {
    const size_t smem = size_t(a.C >> 4) * sizeof(int);
    auto kern = f8_split_kernel<T, NS, AM>;
    if (!allow_smem(reinterpret_cast<const void *>(kern), smem)) return QMV_ERR_CUDA;
    const int64_t blocks = (a.R + T - 1) / T;  // one per tile (split_fits: all resident)
    if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) return QMV_ERR_SHAPE;
    blocks_out = int(blocks);
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(256), smem, s, a));
}

template <bool AM>
qmv_status launch_split(const F8Args &a, cudaStream_t s, int &blocks_out) {
    switch (split_steps(a.C)) {
        case 1: return launch_split_t<8, 1, AM>(a, s, blocks_out);
        case 2: return launch_split_t<4, 2, AM>(a, s, blocks_out);
        default: return launch_split_t<2, 4, AM>(a, s, blocks_out);
    }
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
        // (tile shape from a sweep on 4096 x 4096: at batch 1, 4 rows x 4
        // steps ran 8.2 us against 8.8 us for 2 x 8 and 10.3 us for 2 x 4)
        constexpr int TS = (B == 1) ? 4 : 2, NSTEP = (B == 1) ? 4 : (B <= 2) ? 8 : 4;
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
    if (tc_fits(a, batch)) return launch_tc(a, batch, AM, s, blocks);    // batch 5..8: tcgen05, weights by TMA
    if (mma_fits(a, batch)) return launch_mma(a, batch, AM, s, blocks);  // batch 2..8: mma.sync
    if (fast) {
        switch (batch) {
            case 1:  // few rows of 4096..16384 columns: one wave, columns split over warps
                return split_fits<AM>(a) ? launch_split<AM>(a, s, blocks) : launch_fast<1, AM>(a, s, blocks);
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
}  // namespace f8

qmv_status launch_f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                            int64_t SC, const float *x, int batch, float *y, cudaStream_t s) {
    f8::F8Args a{w, scale, x, y, R, C, SR, SC, nullptr, nullptr, nullptr, nullptr};
    int blocks = 0;
    return f8::launch_any<false>(a, batch, s, blocks);
}

qmv_status launch_f8_matvec_argmax(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                                   int64_t SC, const float *x, int batch, float *y, int64_t *out_index,
                                   float *out_value, void *workspace, int64_t workspace_bytes,
                                   cudaStream_t s) {
    // workspace: the arrival counter in its first 16 bytes, then the partials
    unsigned char *base = static_cast<unsigned char *>(workspace);
    f8::F8Args a{w,     scale, x, y, R, C, SR, SC, reinterpret_cast<f8::ArgBest *>(base + QMV_ARGMAX_COUNTER_BYTES),
                 reinterpret_cast<unsigned *>(base), out_index, out_value};
    // No y, but room behind the partials for the batch's logits: keep them
    // there when that lets the call run on the tcgen05 kernel (which needs y).
    const int64_t off = QMV_F8_ARGMAX_LOGITS_OFFSET(batch);
    if (!y && workspace_bytes - off >= int64_t(batch) * R * 4) {
        f8::F8Args t = a;
        t.y = reinterpret_cast<float *>(base + off);
        if (f8::tc_fits(t, batch)) a.y = t.y;
    }
    int blocks = 0;
    return f8::launch_any<true>(a, batch, s, blocks);
}

}  // namespace qmv
