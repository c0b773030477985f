// f8_mma_kernels.cu -- block-scaled F8 E4M3 matvec at batch 2..8 on the
// tensor cores (mma.sync m16n8k16, f16 operands, float32 accumulation), for
// sm_103a.
//
// Method: ds4f-disk issue #6 "attention + tokenizer + sampling", work item 1
// and step 1 (the F8 E4M3 + E8M0 matvec), work item 3 (the ~246k x 4096 head)
// and step 3 (greedy selection on the head).
//
//   y[v][r] = sum_c E4M3(w[r][c]) * E8M0(scale[r*SR/R][c*SC/C]) * x[v][c]
#include "f8_common.cuh"
#include "mma_device.cuh"

namespace qmv {
namespace f8 {
namespace {

using mma::cp_async_commit;
using mma::cp_async_wait;
using mma::kRing;
using mma::mma_16816;
using mma::split_block;

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
        const float sa = dev::e8m0(st.s[0][k]), sb = dev::e8m0(st.s[1][k]);
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
// Every thread of the block calls it (argmax_complete follows with barriers);
// `scratch` is the kernel's epilogue buffer, idle by then.
__device__ __forceinline__ void mma_argmax_store(float best_v, int64_t best_i, const F8Args &a, int batch,
                                                 void *scratch) {
    const int warp = threadIdx.x >> 5, o = threadIdx.x;
    if (warp < (16 * batch + 31) / 32) {  // warp-uniform
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
    argmax_complete(a, batch, scratch);
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
    if (AM) mma_argmax_store(best_v, best_i, a, batch, red);
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

template <int NJ, int NK, bool AM, bool EARLY>
__global__ void __launch_bounds__(512, 1) f8_mma_staged_kernel(F8Args a, int batch, int div32) {
    constexpr bool kEarly = NJ == 1 || EARLY;  // first tiles issued before the dependency wait
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
    if (kEarly) pdl_trigger();
    for (int kb = threadIdx.x; kb < NW * NK; kb += blockDim.x) cb64[kb] = int((int64_t(kb) * 64 * a.SC) / a.C);

    const int64_t ntiles = (a.R + 15) >> 4;
    const int64_t gstride = gridDim.x;
    // At batch 2-4 (NJ = 1) the first kRing - 1 tiles of weights go out
    // before the dependency wait (they never depend on the preceding kernel).
    // At batch 5-8 (NJ = 2), where the kernel sits at its register limit,
    // only for matrices of a few tiles per block (EARLY): issued early on the
    // head, its batch-8 argmax ran 209 against 203 us, while 4096 x 4096
    // went from 12.1 to 10.8 us.  Otherwise they go out after the barrier.
    if (kEarly && int64_t(blockIdx.x) < ntiles) {  // block-uniform
#pragma unroll
        for (int st = 0; st < kRing - 1; st++) {
            const int64_t tl = blockIdx.x + st * gstride;
            if (tl < ntiles) mma::issue_tile<NK>(ring + uint32_t(st * SLOT), a.w, a.R, a.C, tl, kb_lo, lane);
            cp_async_commit();
        }
    }
    pdl_wait();
    if (!kEarly) pdl_trigger();
    __syncthreads();
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
        if (!kEarly) {
            // the first kRing - 1 tiles go out before the B fragments are built
#pragma unroll
            for (int st = 0; st < kRing - 1; st++) {
                const int64_t tl = blockIdx.x + st * gstride;
                if (tl < ntiles) mma::issue_tile<NK>(ring + uint32_t(st * SLOT), a.w, a.R, a.C, tl, kb_lo, lane);
                cp_async_commit();
            }
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
                const float s_a = dev::e8m0(sa[k]), s_b = dev::e8m0(sb[k]);
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
    if (AM) mma_argmax_store(best_v, best_i, a, batch, red);
}

// The tensor-core kernel: C % 64 == 0 with at least four 64-column blocks
// (one warp per block, and the tile epilogue needs 16 * batch <= 128 threads),
// 16-byte aligned w and x, every 64-column block inside one scale block, and
// its shared memory in reach.
constexpr size_t kMmaSmemMax = 200 * 1024;
// Batch 5-8 matrices of at most this many 16-row tiles per block issue their
// first tiles before the dependency wait (EARLY).
constexpr int64_t kEarlyTilesPerBlock = 8;
bool mma_fits_impl(const F8Args &a, int batch) {
    if (batch < 2 || a.C % 64 != 0 || a.C < 256) return false;
    if (reinterpret_cast<uintptr_t>(a.w) % 16 != 0 || reinterpret_cast<uintptr_t>(a.x) % 16 != 0) return false;
    const int NJ = (batch + 3) / 4;
    const int NW = a.C / 64 < 16 ? int(a.C / 64) : 16;
    if (mma_smem_bytes(a.C, NJ, NW) > kMmaSmemMax) return false;
    return chunks_uniform(a.C, a.SC, 64);
}

template <int NJ, int NK, bool AM, bool EARLY = false>
qmv_status launch_mma_staged(const F8Args &a, int batch, cudaStream_t s, int &blocks_out) {
    const int NW = int(a.C / 64 / NK);
    const size_t smem = mma::staged_smem_bytes(NW, NK, NJ, size_t(NW) * NK * 4);  // + scale columns
    auto kern = f8_mma_staged_kernel<NJ, NK, AM, EARLY>;
    const void *kp = reinterpret_cast<const void *>(kern);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int64_t ntiles = (a.R + 15) / 16;
    int64_t blocks = int64_t(occupancy(kp, 32 * NW, smem)) * sm_count();
    if (blocks > ntiles) blocks = ntiles;
    if (AM && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
    if constexpr (NJ == 2 && !EARLY) {
        if (ntiles <= kEarlyTilesPerBlock * blocks) return launch_mma_staged<NJ, NK, AM, true>(a, batch, s, blocks_out);
    }
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

}  // namespace

bool mma_fits(const F8Args &a, int batch) { return a.R > 0 && mma_fits_impl(a, batch); }

qmv_status launch_mma(const F8Args &a, int batch, bool am, cudaStream_t s, int &blocks_out) {
    if (batch <= 4)
        return am ? launch_mma<1, true>(a, batch, s, blocks_out) : launch_mma<1, false>(a, batch, s, blocks_out);
    return am ? launch_mma<2, true>(a, batch, s, blocks_out) : launch_mma<2, false>(a, batch, s, blocks_out);
}

}  // namespace f8
}  // namespace qmv
