// mma_device.cuh -- device pieces shared by the tensor-core matvec kernels
// (f8_kernels.cu, i8_kernels.cu) for sm_103a: cp.async staging of 8-bit
// weight tiles, the f16 hi/lo split of the activations into mma B fragments,
// mma.sync m16n8k16, and the fixed-order tile epilogue.
//
// Shapes.  A block owns tiles of 16 weight rows in grid-stride order; warp w
// owns NK (1, 2 or 4) 64-column blocks of every tile, starting at column block
// kb_lo = w * NK.  Lane (g = lane/4, t = lane%4) handles rows g and g+8 and the
// 16 bytes at column 64*kb + 16*t of each; mma i (0..3) of a column block binds
// its k slots 2t, 2t+1, 2t+8, 2t+9 to columns 64*kb + 16*t + 4*i + 0, 1, 2, 3 in
// A and B alike (a dot product may be summed in any order).  The 8 columns of
// one mma are (vector, hi | lo) pairs of 4 vectors: vector group j covers
// vectors 4j .. 4j+3, and the lane's accumulators hold rows g, g+8 of vector
// 4j+t as (hi part, lo part).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "device_common.cuh"

namespace qmv {
namespace mma {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRing = 3;  // tiles per warp in the cp.async ring

using dev::cp_async16;
using dev::cp_async_commit;
using dev::cp_async_wait;

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &d, int q) {
    return q == 0 ? d.x : q == 1 ? d.y : q == 2 ? d.z : d.w;
}

// Splits one 64-column block of one activation vector (lane l holds columns
// 2l and 2l+1; the whole warp calls it): with m the block's largest finite
// |x| and E = min(14 - floor(log2 m), 127) (0 when m = 0), x * 2^E = hi + lo,
// hi = f16(x * 2^E), lo = f16(x * 2^E - hi).  Returns the packed f16 pairs
// and f = 2^-E, or f = NaN when the block holds Inf or NaN.
__device__ __forceinline__ void split_block(float2 xv, uint32_t &hi, uint32_t &lo, float &f) {
    const bool fin = isfinite(xv.x) && isfinite(xv.y);
    float m = fmaxf(isfinite(xv.x) ? fabsf(xv.x) : 0.0f, isfinite(xv.y) ? fabsf(xv.y) : 0.0f);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, d));
    const bool all_finite = __all_sync(kFull, fin);
    int E = 0;
    if (m > 0.0f) E = min(14 - ilogbf(m), 127);  // in [-113, 127]
    const float up = __uint_as_float(uint32_t(127 + E) << 23);
    const float down = (E == 127) ? __uint_as_float(0x00400000u) : __uint_as_float(uint32_t(127 - E) << 23);
    const float s0 = xv.x * up, s1 = xv.y * up;
    const __half h0 = __float2half_rn(s0), h1 = __float2half_rn(s1);
    const __half l0 = __float2half_rn(s0 - __half2float(h0)), l1 = __float2half_rn(s1 - __half2float(h1));
    hi = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
    lo = uint32_t(__half_as_ushort(l0)) | (uint32_t(__half_as_ushort(l1)) << 16);
    f = all_finite ? down : __uint_as_float(0x7fc00000u);
}

// This warp's B fragments (column block k of its range, mma i, vector group
// j, register half) and the 2^-E factors of vector 4j+t.
template <int NJ>
struct StagedB {
    uint32_t b[4][4][NJ][2];
    float f[4][NJ];
};

// Builds StagedB for column blocks kb_lo .. kb_lo+nk-1 of the activations,
// whose 16 values at column c0 of vector v come from load16(v, c0, xs).
// Lane (g, t)'s fragments of column block kb all come from its own 16-column
// chunk 64*kb + 16*t of vector 4j + g/2 (hi part for even g, lo for odd g),
// so each lane loads that chunk and splits it itself; the block's largest
// |x| is a max over the 4 lanes t of the same g (two shuffles).  The same
// split as split_block: m, E = min(14 - floor(log2 m), 127), hi, lo, 2^-E
// (NaN when the block holds Inf or NaN).  f of vector 4j+t (the lane's
// accumulator) comes from lane 8t, which split that vector.
template <int NJ, typename Load16>
__device__ __forceinline__ void build_b_from(StagedB<NJ> &B, Load16 load16, int batch, int kb_lo, int nk,
                                             int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        if (k >= nk) break;  // warp-uniform
#pragma unroll
        for (int j = 0; j < NJ; j++) {
            const int v = 4 * j + (g >> 1);
            float xs[16];
            if (v < batch) {
                load16(v, int64_t(kb_lo + k) * 64 + 16 * t, xs);
            } else {
#pragma unroll
                for (int e = 0; e < 16; e++) xs[e] = 0.0f;
            }
            float m = 0.0f;
            int fin = 1;
#pragma unroll
            for (int e = 0; e < 16; e++) {
                const bool f = isfinite(xs[e]);
                fin &= int(f);
                m = fmaxf(m, f ? fabsf(xs[e]) : 0.0f);
            }
            m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
            m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
            fin &= __shfl_xor_sync(kFull, fin, 1);
            fin &= __shfl_xor_sync(kFull, fin, 2);
            int E = 0;
            if (m > 0.0f) E = min(14 - ilogbf(m), 127);  // in [-113, 127]
            const float up = __uint_as_float(uint32_t(127 + E) << 23);
            const float down = (E == 127) ? __uint_as_float(0x00400000u) : __uint_as_float(uint32_t(127 - E) << 23);
            const float f = fin ? down : __uint_as_float(0x7fc00000u);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                uint32_t half2[2];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const float s0 = xs[4 * i + 2 * h] * up, s1 = xs[4 * i + 2 * h + 1] * up;
                    const __half h0 = __float2half_rn(s0), h1 = __float2half_rn(s1);
                    __half o0 = h0, o1 = h1;
                    if (g & 1) {
                        o0 = __float2half_rn(s0 - __half2float(h0));
                        o1 = __float2half_rn(s1 - __half2float(h1));
                    }
                    half2[h] = uint32_t(__half_as_ushort(o0)) | (uint32_t(__half_as_ushort(o1)) << 16);
                }
                B.b[k][i][j][0] = half2[0];
                B.b[k][i][j][1] = half2[1];
            }
            B.f[k][j] = __shfl_sync(kFull, f, 8 * t);
        }
    }
}

// StagedB from float activations x [batch, C].
template <int NJ>
__device__ __forceinline__ void build_b(StagedB<NJ> &B, const float *x, int64_t C, int batch, int kb_lo, int nk,
                                        int lane) {
    auto load16 = [&](int v, int64_t c0, float (&xs)[16]) {
        const float4 *src = reinterpret_cast<const float4 *>(x + int64_t(v) * C + c0);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float4 f4 = __ldg(src + q);
            xs[4 * q] = f4.x;
            xs[4 * q + 1] = f4.y;
            xs[4 * q + 2] = f4.z;
            xs[4 * q + 3] = f4.w;
        }
    };
    build_b_from<NJ>(B, load16, batch, kb_lo, nk, lane);
}

// Copies this warp's part of tile `tl` of the byte matrix w [R, C] -- 16 rows
// x NK 64-column blocks from column 64*kb_lo, rows past R clamped to R-1 --
// into the stage at shared address `dst`.  The copies are coalesced (lane l of
// copy m takes 16-byte chunk e = 32m + l, row e / (4 NK), so each instruction
// reads whole 128-byte lines); chunk c of row rho is stored at position
// c ^ (rho & 7) (mod 4 NK) of the row, which makes the fragment-order reads
// of row_chunk() conflict free.  Requires C <= 4096 (rho * C fits in 32 bits).
template <int NK>
__device__ __forceinline__ void issue_tile(uint32_t dst, const uint8_t *w, int64_t R, int64_t C, int64_t tl,
                                           int kb_lo, int lane) {
    constexpr int NCH = 4 * NK;  // 16-byte chunks per row
    constexpr int LOG = NK == 1 ? 2 : NK == 2 ? 3 : 4;
    const int64_t r0 = tl * 16;
    const uint8_t *base = w + r0 * C + int64_t(kb_lo) * 64;
    const bool full = r0 + 16 <= R;  // block-uniform: only the last tile is ragged
    const int C32 = int(C);
#pragma unroll
    for (int m = 0; m < NCH / 2; m++) {
        const int e = 32 * m + lane, rho = e >> LOG, c = e & (NCH - 1);
        const int rr = full ? rho : int(min(int64_t(rho), R - 1 - r0));
        const int pos = c ^ (rho & (NCH - 1) & 7);
        cp_async16(dst + uint32_t((rho * NCH + pos) * 16), base + (rr * C32 + 16 * c));
    }
}

// The 16 bytes of row `rho` at chunk c (= 4k + t) of a stage written by
// issue_tile<NK>.
template <int NK>
__device__ __forceinline__ uint4 row_chunk(const uint4 *stage, int rho, int c) {
    constexpr int NCH = 4 * NK;
    return stage[rho * NCH + (c ^ (rho & (NCH - 1) & 7))];
}

// Tile epilogue.  Every warp stores its partial sums (rows g and g+8 of
// vector 4j+t) to red[buf]; after the barrier, reducer thread o = 16*v + rho
// adds the warps' partials for row r0+rho of vector v in a fixed order,
// replaces a non-finite result by exact(row, v) (a warp-collective exact
// evaluation), stores it to y [batch, R] when y is not NULL, and, with AM,
// keeps the best (value, row) it has seen by arg_better.  Every thread of the
// block calls it.
template <int NJ, bool AM, typename Exact, typename Better>
__device__ __forceinline__ void tile_epilogue(float (&tot)[NJ][2], float *red, int buf, int NW, int batch,
                                              int64_t R, float *y, int64_t r0, float &best_v, int64_t &best_i,
                                              Exact exact, Better better) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2 *rw = reinterpret_cast<float2 *>(red) + ((buf * NW + warp) * NJ) * 32;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        rw[j * 32 + lane] = make_float2(tot[j][0], tot[j][1]);
        tot[j][0] = tot[j][1] = 0.0f;
    }
    __syncthreads();
    if (warp < (16 * batch + 31) / 32) {  // warp-uniform
        const int o = threadIdx.x, o_v = o >> 4, o_rho = o & 15;
        const bool valid = o < 16 * batch && r0 + o_rho < R;
        float sum = 0.0f;
        if (valid) {
            const int j = o_v >> 2, lp = (o_rho & 7) * 4 + (o_v & 3), comp = o_rho >> 3;
            // four interleaved partial sums, combined in a fixed order
            const float *rp = red + ((buf * NW * NJ + j) * 32 + lp) * 2 + comp;
            const int wstride = NJ * 64;
            float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
            int w2 = 0;
            for (; w2 + 4 <= NW; w2 += 4) {
                p0 += rp[(w2 + 0) * wstride];
                p1 += rp[(w2 + 1) * wstride];
                p2 += rp[(w2 + 2) * wstride];
                p3 += rp[(w2 + 3) * wstride];
            }
            for (; w2 < NW; w2++) p0 += rp[w2 * wstride];
            sum = (p0 + p1) + (p2 + p3);
        }
        unsigned bad = __ballot_sync(kFull, valid && !isfinite(sum));
        while (bad) {
            const int bl = __ffs(bad) - 1;
            bad &= bad - 1;
            const int ob = warp * 32 + bl;
            const float ex = exact(r0 + (ob & 15), ob >> 4);
            if (lane == bl) sum = ex;
        }
        if (valid) {
            if (AM && better(sum, r0 + o_rho, best_v, best_i)) {
                best_v = sum;
                best_i = r0 + o_rho;
            }
            if (y) y[int64_t(o_v) * R + r0 + o_rho] = sum;
        }
    }
}

// Host side.  The staged kernels give every warp NK = 4, 2 or 1 whole
// 64-column blocks: the largest that divides C / 64 with at most 16 warps and
// at least ceil(batch / 2) (the tile epilogue has 16 * batch reducer
// threads).  0: not applicable.
inline int staged_nk(int64_t C, int batch) {
    if (C % 64 != 0 || C < 64) return 0;
    const int64_t nkb = C / 64;
    for (int nk = 4; nk >= 1; nk >>= 1)
        if (nkb % nk == 0 && nkb / nk <= 16 && nkb / nk >= (batch + 1) / 2) return nk;
    return 0;
}

// Shared memory of a staged kernel with NW warps: the cp.async rings, the
// double-buffered partial sums, and `extra` bytes after them.
inline size_t staged_smem_bytes(int NW, int NK, int NJ, size_t extra) {
    return size_t(NW) * kRing * 16 * 4 * NK * 16 + size_t(2) * NW * NJ * 32 * 8 + extra;
}

}  // namespace mma
}  // namespace qmv
