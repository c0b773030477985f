// f8_tc_kernels.cu -- block-scaled F8 E4M3 matvec at batch 5..8 on the
// fifth-generation tensor cores (tcgen05.mma kind::f8f6f4, accumulators in
// tensor memory, weights streamed by TMA), for sm_103a.
//
// Method: ds4f-disk issue #6 "attention + tokenizer + sampling", work item 1
// and step 1 (the F8 E4M3 + E8M0 matvec), work item 3 (the ~246k x 4096 head)
// and step 3 (greedy selection on the head).
//
//   y[v][r] = sum_c E4M3(w[r][c]) * E8M0(scale[r*SR/R][c*SC/C]) * x[v][c]
//
// Orientation.  A tcgen05.mma costs about the same whatever its N (16 .. 256),
// so the weights go in as the wide operand: N = 256 weight rows of one tile,
// read by the tensor core straight from the TMA ring as raw E4M3 bytes (no
// decode on the CUDA cores).  The activations are the M = 128 operand, of
// which 8 rows per vector slot are used: vector v's piece p sits in row 8v + p.
//
// Pieces.  Per vector v and 128-column block kb, with m the largest finite |x|
// there and E = 7 - floor(log2 m), x * 2^E lies below 256 and is split into
// eight E4M3 pieces: piece 0 = E4M3(x 2^E), and piece p + 1 = E4M3 of 16 times
// the residual left by pieces 0..p, so x * 2^E = sum_p piece_p * 2^-4p.  Each
// piece keeps 4 significant bits of what is left (fewer while it is an E4M3
// subnormal), so an element keeps 2^-16 of itself, or 2^-45 of the block's
// largest |x| (the last piece's subnormal step) if that is larger; elements
// within 2^-21 of the largest are split exactly.  E4M3 x E4M3 products are
// exact in the float32 accumulator.
//
// Passes.  Up to 4 vectors (32 piece rows) the pieces of all of K take 128 KB
// of shared memory; 5..8 vectors (64 rows) take twice that, so the
// K range runs in two passes of half the blocks each, the second adding onto
// the partial sums the first stored in y (the same thread reads back what it
// wrote, so the result is deterministic).
//
// Scales.  Every 128-column block must lie in one scale column block and
// every 64-row unit in one scale row (each scale block starts on a multiple of
// 128 columns and of 64 rows), so within a tile's unit the factor
// 2^(s - 127) * 2^-(E + 4p) of accumulator row 8v + p and block kb is one
// power of two.  Each block gets a fresh accumulator D (4 MMAs of K = 32); the
// epilogue warps read D back (tcgen05.ld), multiply row 8v + p by its factor
// and add into registers -- relative to a reference exponent per vector (its
// first nonzero block's), so that tiny or huge x does not push the factors
// out of float range; the sum is scaled back once at the end.  At the end of a tile the 8 pieces of each vector
// (lanes 8v' .. 8v' + 7 of a warp) are summed by three exchange rounds.
//
// Warps (512 threads, one block per SM): warp 2 issues the TMA copies (lane
// 0), warp 3 issues the MMAs (lane 0) and owns the tensor memory, the warps
// 0 mod 4 (and 1 mod 4 at 5..8 vectors) are the epilogue -- a warp reads the
// TMEM lanes of its number mod 4, and piece rows 32q .. 32q + 31 hold vectors
// 4q .. 4q + 3 -- and the rest build the activation pieces, block by block,
// each block announced on its own mbarrier so the MMAs start on block 0 at
// once.  A block's rows are 64-row units [u0, u1) of the matrix, in tiles of
// up to four units; the TMA loads one 64-row box per unit, so a short last
// tile costs only its own rows.
//
// Memory.  Shared: the pieces of one pass (128 KB), a ring of three 32 KB
// weight stages (256 rows x 128 bytes, 128-byte swizzle), the scale column of
// every block, the block exponents and the barriers -- 226 KB at C = 4096.
// A pass after the first rebuilds each slot of pieces as soon as the previous
// pass's last MMAs on it are done, so the next pass starts without a pause.
// Tensor memory: two 256-column accumulators.
//
// Fix-up.  A result that is not finite (an E4M3 code 0x7F / 0xFF, which the
// tensor core reads as NaN; a NaN scale; Inf or NaN in x, which marks its
// block; an overflow) is recomputed by the exact per-element path, which gives
// those inputs their per-element meaning.
//
// Waits.  Every mbarrier wait gives up after one second (%globaltimer): the
// role then stops, its results are not valid, and the library's count of
// abandoned waits (qmv_tc_wait_timeouts) goes up.  No wait is expected to
// run out; the limit keeps a fault elsewhere from hanging the GPU.
#include <cuda.h>

#include <mutex>

#include "f8_common.cuh"

namespace qmv {
namespace f8 {

// Waits abandoned after their time limit, summed over all calls (read by
// qmv_tc_wait_timeouts).
__device__ unsigned long long g_tc_timeouts = 0;

namespace {

constexpr int kTcThreads = 512;
constexpr int kTcRows = 256, kTcUnit = 64, kTcChunk = 128;       // tile rows, unit rows, K-block columns
constexpr int kTcStageBytes = kTcRows * kTcChunk;                // 32 KB: one tile x one K-block
constexpr int kTcUnitBytes = kTcUnit * kTcChunk;                 // 8 KB: one TMA box
constexpr int kTcStages = 3;
constexpr int kTcND = 2;                                         // accumulators of 256 columns
constexpr int kTcTmemCols = 512;
constexpr int kTcPieces = 8;                                     // E4M3 pieces per vector
constexpr int kTcMaxJobs = 4;                                    // K-blocks per building warp and pass
constexpr int kWTma = 2, kWMma = 3;                              // (warps 0, 1 mod 4 may be epilogue)
constexpr int kEZero = 100000, kENonFinite = 100001;             // block exponent markers
constexpr uint64_t kWaitNs = 1000000000ull;                      // one second
constexpr int kTcMinUnitsPerSm = 3;                              // smaller matrices: the mma.sync kernel

// Vector slots (rows 8v + p of the pieces): 4 at batch <= 4, else 8; the K
// range then runs in one pass or two, so the pieces of one pass fit 128 KB.
__host__ __device__ inline int tc_slots(int batch) { return batch <= 4 ? 4 : 8; }
__host__ __device__ inline int tc_passes(int nv) { return nv / 4; }
__host__ __device__ inline int pass_blocks(int nkb, int passes) { return (nkb + passes - 1) / passes; }
// Warps that build pieces: all but the TMA and MMA warps and the epilogue warps.
__host__ __device__ inline int tc_build_warps(int nv) { return kTcThreads / 32 - 2 - 4 * (nv / 4); }

__host__ __device__ inline size_t tc_smem_bytes(int64_t C, int nv) {
    const int64_t nkb = C / kTcChunk, nkbp = pass_blocks(int(nkb), tc_passes(nv));
    return size_t(1024                                       // alignment of the base to 1024
                  + nkbp * 8 * nv * kTcPieces * 16           // pieces of one pass
                  + int64_t(kTcStages) * kTcStageBytes       // weight ring
                  + nkb * 4 + nkb * 32                       // scale columns, block exponents
                  + 8 * (2 * kTcStages + 2 * kTcND + 1 + 2 * nkbp) + 16);  // barriers, TMEM address
}

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return uint32_t(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ bool bar_wait_slow(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 64; i++)
            if (bar_try(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) {
            atomicAdd(&g_tc_timeouts, 1ull);
            return false;
        }
    }
}
// Waits for the phase of `bar` with this parity; false after the time limit.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
    return bar_try(bar, parity) || bar_wait_slow(bar, parity);
}
__device__ __forceinline__ void bar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// One 64-row x 128-byte box of the weights (x = column byte, y = row), marked
// first to leave L2 (the weights are read once per call).
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D (tmem) [+]= A (smem) x B (smem), E4M3 operands, float32 accumulator.
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// Shared-memory operand descriptors (sm_100 format: start, leading and
// stride byte offsets >> 4, version 1 at bit 46, layout at bits 61..63).
// Pieces: no swizzle, K-major, 8-row x 16-byte cores; K-adjacent cores
// `core_bytes` apart (all piece rows of one 16-column core), M-adjacent 128
// bytes apart.  Rows past the pieces of the M = 128 operand read the next
// cores (unused accumulator rows).
__device__ __forceinline__ uint64_t piece_desc(uint32_t saddr, uint32_t core_bytes) {
    return uint64_t((saddr & 0x3FFFF) >> 4) | (uint64_t((core_bytes & 0x3FFFF) >> 4) << 16) | (uint64_t(128 >> 4) << 32) |
           (uint64_t(1) << 46);
}
// Weights: 128-byte swizzle, K-major (rows of 128 bytes, 8-row groups 1024
// bytes apart), as the TMA writes them.
__device__ __forceinline__ uint64_t weight_desc(uint32_t saddr) {
    return uint64_t((saddr & 0x3FFFF) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) |
           (uint64_t(2) << 61);
}
// Instruction descriptor: float32 D, E4M3 A and B (both K-major), N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(256 >> 3) << 17) | (uint32_t(128 >> 4) << 24);

// Two floats -> an E4M3 pair, rounded to nearest even (`a` in the low byte).
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}
__device__ __forceinline__ float2 from_e4m3x2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two)));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// 2^(s - 127) * 2^-(E - E0 + 4p) as float32: the factor of accumulator row
// 8v + p for a block with scale code s and exponent E, relative to the
// vector's reference exponent E0 (the result is scaled by 2^-E0 at the end).
// A power of two; 0 below 2^-149, Inf above float range, NaN for a NaN scale
// or a non-finite block.
__device__ __forceinline__ float block_factor(unsigned s, int E, int E0, int p) {
    if (E == kENonFinite || s == 255u) return __uint_as_float(0x7fc00000u);
    if (E == kEZero) return 0.0f;
    const int ex = int(s) - 127 - (E - E0) - 4 * p;
    return ex > 127 ? __uint_as_float(0x7f800000u)
         : ex >= -126 ? __uint_as_float(uint32_t(ex + 127) << 23)
         : ex >= -149 ? __uint_as_float(1u << (ex + 149)) : 0.0f;
}

// The exact per-element path for the results of an epilogue warp that are
// not finite (warp-collective; lane l holds vector 4q + l / 8 and the 8 rows
// r0 + c0(l % 8) + j).  Out of line: it is rare and would crowd the registers
// of the epilogue.
struct Z8 {
    float z[8];
};
__device__ __noinline__ Z8 fix_nonfinite(const F8Args &a, Z8 zz, bool live, int nr, int64_t r0, int q) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        unsigned bad = __ballot_sync(kFull, live && j < nr && !isfinite(zz.z[j]));
        while (bad) {
            const int bl = __ffs(bad) - 1;
            bad &= bad - 1;
            const int pb = bl & 7;
            const int cb = 32 * (pb & 1) + 16 * ((pb >> 1) & 1) + 8 * (pb >> 2);
            const float ex = f8_row_exact(a, r0 + cb + j, 4 * q + (bl >> 3), nullptr);
            if (lane == bl) zz.z[j] = ex;
        }
    }
    return zz;
}

template <bool AM>
__global__ void __launch_bounds__(kTcThreads, 1) f8_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ F8Args a, int batch) {
    extern __shared__ unsigned char tc_smem[];
    const uint32_t raw0 = smem_u32(tc_smem);
    const uint32_t base = (raw0 + 1023u) & ~1023u;
    unsigned char *sm = tc_smem + (base - raw0);
    const int nv = tc_slots(batch), passes = tc_passes(nv);  // vector slots, passes over K
    const int nkb = int(a.C / kTcChunk), nkbp = pass_blocks(nkb, passes);
    const uint32_t core_bytes = uint32_t(nv) * kTcPieces * 16;  // one 16-column core of every piece row
    const uint32_t blk_bytes = 8 * core_bytes;                   // one 128-column block of pieces
    const uint32_t s_ring = base + uint32_t(nkbp) * blk_bytes;   // (the pieces' unused rows read into it)
    int *cbk = reinterpret_cast<int *>(sm + (s_ring - base) + kTcStages * kTcStageBytes);
    int *eb = cbk + nkb;  // [kb][8] block exponents
    const uint32_t s_bars = (smem_u32(eb + nkb * 8) + 7u) & ~7u;
    const uint32_t full0 = s_bars, empty0 = full0 + 8 * kTcStages, dfull0 = empty0 + 8 * kTcStages,
                   dempty0 = dfull0 + 8 * kTcND, done_bar = dempty0 + 8 * kTcND, ready0 = done_bar + 8,
                   free0 = ready0 + 8 * nkbp;  // free0: [nkbp] slot kbl's pieces no longer read
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + (free0 + 8 * nkbp - base));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarters = nv / 4;  // TMEM lane quarters holding piece rows (rows 8v + p)
    const bool epilogue = (warp & 3) < quarters;
    const int64_t units = (a.R + kTcUnit - 1) / kTcUnit;
    const int64_t u0 = int64_t(blockIdx.x) * units / gridDim.x, u1 = int64_t(blockIdx.x + 1) * units / gridDim.x;
    auto kb_begin = [&](int pass) { return pass * nkb / passes; };
    // phase parity of slot kbl's readiness barrier in `pass`: its uses by earlier passes
    auto ready_parity = [&](int pass, int kbl) {
        uint32_t uses = 0;
        for (int p2 = 0; p2 < pass; p2++) uses += kbl < kb_begin(p2 + 1) - kb_begin(p2) ? 1u : 0u;
        return uses & 1u;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; i++) {
            bar_init(full0 + 8 * i, 1);
            bar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < kTcND; i++) {
            bar_init(dfull0 + 8 * i, 1);
            bar_init(dempty0 + 8 * i, 4 * quarters);
        }
        bar_init(done_bar, 1);
        for (int i = 0; i < nkbp; i++) {
            bar_init(ready0 + 8 * i, 1);
            bar_init(free0 + 8 * i, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTcTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    for (int kb = threadIdx.x; kb < nkb; kb += blockDim.x) cbk[kb] = int((int64_t(kb) * kTcChunk * a.SC) / a.C);
    pdl_trigger();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_holder;

    float best_v = -INFINITY;  // argmax: the best of this thread's rows
    int64_t best_i = INT64_MAX;

    if (warp == kWTma) {
        // ---- producer: stage g holds K-block kb of the tile's units, one box per unit.
        // The weights are read-only for the library's calls, so the copies start
        // before the dependency wait.
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
            uint32_t g = 0;
            bool ok = true;
            for (int pass = 0; pass < passes && ok; pass++)
                for (int64_t ut = u0; ut < u1 && ok; ut += 4) {
                    const int nu = int(min(int64_t(4), u1 - ut));
                    for (int kb = kb_begin(pass); kb < kb_begin(pass + 1); kb++, g++) {
                        const uint32_t s = g % kTcStages, u = g / kTcStages;
                        if (u > 0 && !bar_wait(empty0 + 8 * s, (u - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        bar_expect_tx(full0 + 8 * s, uint32_t(nu * kTcUnitBytes));
                        for (int i = 0; i < nu; i++)
                            tma_load(s_ring + s * kTcStageBytes + i * kTcUnitBytes, &wmap, kb * kTcChunk,
                                     int((ut + i) * kTcUnit), full0 + 8 * s);
                    }
                }
            // the copies still in flight land before the block can exit
            for (uint32_t k = g > uint32_t(kTcStages) ? g - kTcStages : 0; k < g; k++)
                bar_wait(full0 + 8 * (k % kTcStages), (k / kTcStages) & 1);
        }
        __syncwarp();
        pdl_wait();  // (the argmax completion below reads other blocks' results)
    } else if (warp == kWMma) {
        pdl_wait();
        // ---- MMA issuer: per stage, four K = 32 steps into a fresh accumulator
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int pass = 0; pass < passes && ok; pass++) {
                for (int64_t ut = u0; ut < u1 && ok; ut += 4)
                    for (int kb = kb_begin(pass); kb < kb_begin(pass + 1); kb++, g++) {
                        const int kbl = kb - kb_begin(pass);
                        const uint32_t s = g % kTcStages, u = g / kTcStages, d = g % kTcND, ud = g / kTcND;
                        if ((ut == u0 && !bar_wait(ready0 + 8 * kbl, ready_parity(pass, kbl))) ||
                            !bar_wait(full0 + 8 * s, u & 1) || (ud > 0 && !bar_wait(dempty0 + 8 * d, (ud - 1) & 1))) {
                            ok = false;
                            break;
                        }
                        tc_after();
#pragma unroll
                        for (int kk = 0; kk < 4; kk++)
                            tc_mma(tmem + d * 256, piece_desc(base + uint32_t(kbl) * blk_bytes + uint32_t(2 * kk) * core_bytes, core_bytes),
                                   weight_desc(s_ring + s * kTcStageBytes + kk * 32), kIdesc, kk > 0 ? 1u : 0u);
                        tc_commit(dfull0 + 8 * d);  // the accumulator is ready ...
                        tc_commit(empty0 + 8 * s);  // ... and the stage free, once these MMAs are done
                        // the slot's pieces may be rebuilt for the next pass once the last tile's
                        // MMAs on it are done
                        if (ut + 4 >= u1 && pass + 1 < passes) tc_commit(free0 + 8 * kbl);
                    }
            }
            tc_commit(done_bar);
            bar_wait(done_bar, 0);
        }
        __syncwarp();
    } else if (epilogue) {
        pdl_wait();
        // ---- epilogue: warp (quarter q, slice e) reads TMEM lanes 32q .. 32q + 31 (piece
        // rows of vectors 4q .. 4q + 3) and accumulator columns 64e .. 64e + 63 (unit e of
        // the tile); lane l holds vector 4q + l / 8, piece l % 8
        const int q = warp & 3, e = warp >> 2;
        const int v = 4 * q + (lane >> 3), p = lane & 7;
        const uint32_t t_lane = tmem + (uint32_t(32 * q) << 16);
        // the vector's reference exponent: the first nonzero finite block's E.  Factors
        // relative to it stay in float range unless the vector's blocks differ by ~2^100.
        int e0 = kEZero;
        uint32_t g = 0;
        bool ok = true;
        for (int pass = 0; pass < passes && ok; pass++) {
            const bool last = pass == passes - 1;
            for (int64_t ut = u0; ut < u1 && ok; ut += 4) {
                const bool mine = ut + e < u1;
                const int64_t r0 = (ut + e) * kTcUnit;
                const int64_t srow = mine ? (r0 * a.SR / a.R) * a.SC : 0;
                float acc[64];
#pragma unroll
                for (int j = 0; j < 64; j++) acc[j] = 0.f;
                for (int kb = kb_begin(pass); kb < kb_begin(pass + 1); kb++, g++) {
                    const uint32_t d = g % kTcND, ud = g / kTcND;
                    const int kbl = kb - kb_begin(pass);
                    // every lane waits; the warp goes on only if all of them saw the phase.  The
                    // block's factor is formed while the accumulator is still being computed.
                    const bool ready = ut != u0 || bar_wait(ready0 + 8 * kbl, ready_parity(pass, kbl));
                    float fs = 0.f;
                    if (mine && v < batch && ready) {
                        const int E = eb[kb * 8 + v];
                        if (e0 == kEZero && E != kEZero && E != kENonFinite) e0 = E;
                        fs = block_factor(__ldg(a.scale + srow + cbk[kb]), E, e0 == kEZero ? 0 : e0, p);
                    }
                    const bool seen = ready && bar_wait(dfull0 + 8 * d, ud & 1);
                    if (!__all_sync(kFull, seen)) {
                        ok = false;
                        break;
                    }
                    tc_after();
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        uint32_t dv[32];
                        tc_ld32(t_lane + d * 256 + 64 * e + 32 * h, dv);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                        for (int j = 0; j < 32; j++) acc[32 * h + j] = fmaf(__uint_as_float(dv[j]), fs, acc[32 * h + j]);
                    }
                    tc_before();
                    __syncwarp();
                    if (lane == 0) bar_arrive(dempty0 + 8 * d);
                }
                if (!ok || !mine) continue;  // warp-uniform
                // the eight pieces of vector v sit in lanes 8(v - 4q) .. + 7: three exchange
                // rounds sum them and leave lane (v, p) with the 8 columns c0 .. c0 + 7 of the
                // unit; every column gets ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7))
                float u[32];
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const float send = (p & 1) ? acc[j] : acc[32 + j];
                    const float keep = (p & 1) ? acc[32 + j] : acc[j];
                    u[j] = keep + __shfl_xor_sync(kFull, send, 1);
                }
                float t[16];
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const float send = (p & 2) ? u[j] : u[16 + j];
                    const float keep = (p & 2) ? u[16 + j] : u[j];
                    t[j] = keep + __shfl_xor_sync(kFull, send, 2);
                }
                float z[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float send = (p & 4) ? t[j] : t[8 + j];
                    const float keep = (p & 4) ? t[8 + j] : t[j];
                    z[j] = keep + __shfl_xor_sync(kFull, send, 4);
                }
                const int c0 = 32 * (p & 1) + 16 * ((p >> 1) & 1) + 8 * (p >> 2);
                const int nr = int(min(int64_t(kTcUnit), a.R - r0)) - c0;  // this lane's rows: j < nr
                const bool live = v < batch;
                if (e0 != kEZero) {  // back from the reference exponent: 2^-e0 in two exact steps
                    const int s1 = -e0 < -126 ? -126 : (-e0 > 127 ? 127 : -e0), s2 = -e0 - s1;
                    const float f1 = __uint_as_float(uint32_t(127 + s1) << 23), f2 = __uint_as_float(uint32_t(127 + s2) << 23);
#pragma unroll
                    for (int j = 0; j < 8; j++) z[j] = (z[j] * f1) * f2;
                }
                float *yr = a.y ? a.y + int64_t(v) * a.R + r0 + c0 : nullptr;
                if (pass > 0 && live) {  // earlier passes' sums, stored by this same thread
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        if (j < nr) z[j] = yr[j] + z[j];
                }
                if (last) {
                    // results that are not finite take the exact per-element path (warp-collective)
                    bool any_bad = false;
#pragma unroll
                    for (int j = 0; j < 8; j++) any_bad |= live && j < nr && !isfinite(z[j]);
                    if (__any_sync(kFull, any_bad)) {
                        Z8 zz;
#pragma unroll
                        for (int j = 0; j < 8; j++) zz.z[j] = z[j];
                        zz = fix_nonfinite(a, zz, live, nr, r0, q);
#pragma unroll
                        for (int j = 0; j < 8; j++) z[j] = zz.z[j];
                    }
                }
                if (live) {
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        if (j < nr) {
                            if (yr) yr[j] = z[j];
                            if (AM && last && arg_better(z[j], r0 + c0 + j, best_v, best_i)) {
                                best_v = z[j];
                                best_i = r0 + c0 + j;
                            }
                        }
                    }
                }
            }
        }
        if (AM) {  // the best of vector v over its eight lanes
#pragma unroll
            for (int dd = 1; dd <= 4; dd <<= 1) {
                const float ov = __shfl_xor_sync(kFull, best_v, dd);
                const int64_t oi = __shfl_xor_sync(kFull, best_i, dd);
                if (arg_better(ov, oi, best_v, best_i)) {
                    best_v = ov;
                    best_i = oi;
                }
            }
        }
    } else {
        pdl_wait();
        // ---- activation pieces, K-block by K-block, in the warps with no other role:
        // lane (v = lane % 8, cq = lane / 8) of the warp that owns block kb handles its
        // 16-column cores cq and cq + 4 of vector v.  Piece p of vector v goes to row
        // 8v + p; vectors past the batch are zero.  Each block is announced on its own
        // barrier, so the MMAs start on a pass's first block while later ones are still
        // built; a pass after the first waits until the MMAs are done with the last one.
        int wi = 0, nbuild = 0;  // this warp's index among the building warps, and their number
        for (int w2 = 0; w2 < kTcThreads / 32; w2++) {
            const bool builds = w2 != kWTma && w2 != kWMma && (w2 & 3) >= quarters;
            if (builds && w2 < warp) wi++;
            nbuild += builds ? 1 : 0;
        }
        const int vv = lane & 7, cq = lane >> 3;
        bool ok = u0 < u1;  // (every block has rows: the grid is never wider than the units)
        for (int pass = 0; pass < passes && ok; pass++) {
            const int kb0 = kb_begin(pass), nb = kb_begin(pass + 1) - kb0;
#pragma unroll 1
            for (int half = 0; half < kTcMaxJobs / 2; half++) {
                float4 xs[2][8];
#pragma unroll
                for (int jj = 0; jj < 2; jj++) {
                    const int kbl = wi + (2 * half + jj) * nbuild;
#pragma unroll
                    for (int h = 0; h < 2; h++)
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            xs[jj][4 * h + i] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (kbl < nb && vv < batch)
                                xs[jj][4 * h + i] = __ldg(reinterpret_cast<const float4 *>(
                                                              a.x + int64_t(vv) * a.C + int64_t(kb0 + kbl) * kTcChunk +
                                                              (cq + 4 * h) * 16) + i);
                        }
                }
#pragma unroll
                for (int jj = 0; jj < 2; jj++) {
                    const int kbl = wi + (2 * half + jj) * nbuild;
                    if (kbl >= nb || !ok) break;  // warp-uniform
                    // a slot the previous pass used: wait until its last MMAs are done (passes <= 2)
                    if (pass > 0 && kbl < kb_begin(pass) - kb_begin(pass - 1) &&
                        !__all_sync(kFull, bar_wait(free0 + 8 * kbl, 0))) {
                        ok = false;
                        break;
                    }
                    float r[32];
                    bool fin = true;
                    float m = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float4 t4 = xs[jj][i];
                        r[4 * i] = t4.x;
                        r[4 * i + 1] = t4.y;
                        r[4 * i + 2] = t4.z;
                        r[4 * i + 3] = t4.w;
                    }
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const bool f = isfinite(r[i]);
                        fin &= f;
                        if (!f) r[i] = 0.f;
                        m = fmaxf(m, fabsf(r[i]));
                    }
                    m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
                    const int E = m > 0.f ? 7 - ilogbf(m) : kEZero;  // in [-120, 156]
                    if (m > 0.f) {
                        const int E1 = E > 127 ? 127 : E, E2 = E - E1;  // x * 2^E in two exact steps
                        const float f1 = __uint_as_float(uint32_t(127 + E1) << 23),
                                    f2 = __uint_as_float(uint32_t(127 + E2) << 23);
#pragma unroll
                        for (int i = 0; i < 32; i++) r[i] = r[i] * f1 * f2;
                    }
                    unsigned char *blk = sm + uint32_t(kbl) * blk_bytes;
#pragma unroll
                    for (int pc = 0; pc < kTcPieces; pc++) {
                        uint32_t wv[8];
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            const uint32_t two = to_e4m3x2(r[2 * i], r[2 * i + 1]);
                            if (i & 1) wv[i >> 1] |= two << 16;
                            else wv[i >> 1] = two;
                            if (pc + 1 < kTcPieces) {  // the residual, times 16 (exact)
                                const float2 qv = from_e4m3x2(two);
                                r[2 * i] = (r[2 * i] - qv.x) * 16.f;
                                r[2 * i + 1] = (r[2 * i + 1] - qv.y) * 16.f;
                            }
                        }
                        if (vv < nv) {
                            const int mrow = kTcPieces * vv + pc;
                            const uint32_t roff = uint32_t(mrow >> 3) * 128 + uint32_t(mrow & 7) * 16;
                            *reinterpret_cast<uint4 *>(blk + uint32_t(cq) * core_bytes + roff) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                            *reinterpret_cast<uint4 *>(blk + uint32_t(cq + 4) * core_bytes + roff) =
                                make_uint4(wv[4], wv[5], wv[6], wv[7]);
                        }
                    }
                    const unsigned bad = __ballot_sync(kFull, !fin);  // lanes v, v+8, v+16, v+24 hold vector v
                    if (cq == 0) eb[(kb0 + kbl) * 8 + vv] = ((bad >> vv) & 0x01010101u) ? kENonFinite : E;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // pieces -> tensor core reads
                    __syncwarp();
                    if (lane == 0) bar_arrive(ready0 + 8 * kbl);
                }
            }
        }
    }
    tc_before();
    __syncthreads();
    if (warp == kWMma) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols));
    }
    if (AM) {
        // the block's best per vector from the epilogue warps (the ring is idle now):
        // lane 8k of a quarter-q warp holds vector 4q + k
        ArgBest *wb = reinterpret_cast<ArgBest *>(sm + (s_ring - base));  // [4 slices][8 vectors]
        if (epilogue && (lane & 7) == 0) {
            ArgBest r;
            r.v = best_v;
            r.pad = 0;
            r.i = best_i;
            wb[(warp >> 2) * 8 + 4 * (warp & 3) + (lane >> 3)] = r;
        }
        __syncthreads();
        if (int(threadIdx.x) < batch) {
            const int k = threadIdx.x;
            float bv = wb[k].v;
            int64_t bi = wb[k].i;
            for (int w2 = 1; w2 < 4; w2++)
                if (arg_better(wb[w2 * 8 + k].v, wb[w2 * 8 + k].i, bv, bi)) {
                    bv = wb[w2 * 8 + k].v;
                    bi = wb[w2 * 8 + k].i;
                }
            ArgBest r;
            r.v = bv;
            r.pad = 0;
            r.i = bi;
            a.ws[int64_t(blockIdx.x) * batch + k] = r;
        }
        argmax_complete(a, batch, sm + (s_ring - base) + 1024);
    }
}

// ---- host ---------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, fetched through the runtime (no link against the
// driver library); NULL when the driver does not offer it.
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        (void)cudaGetLastError();
    });
    return fn;
}

// The weights as a 2-D tensor of bytes [R][C], read in 64-row x 128-byte
// boxes with the 128-byte swizzle the MMA descriptors expect.
bool weight_map(const F8Args &a, CUtensorMap &map) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(a.C), cuuint64_t(a.R)};
    const cuuint64_t strides[1] = {cuuint64_t(a.C)};
    const cuuint32_t box[2] = {kTcChunk, kTcUnit};
    const cuuint32_t elem[2] = {1, 1};
    return enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.w), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_fits(const F8Args &a, int batch) {
    // batch 5..8: at 2..4 vectors the mma.sync kernels measured as fast or
    // faster (the layout below serves them, but is not routed to)
    if (batch < 5 || batch > 8 || a.R < 1 || a.R > (int64_t(1) << 31) - 1) return false;
    // enough rows for every block to stream a while: the activation pieces are
    // built once per block, which smaller matrices do not repay
    if ((a.R + kTcUnit - 1) / kTcUnit < int64_t(kTcMinUnitsPerSm) * sm_count()) return false;
    const int nv = tc_slots(batch), passes = tc_passes(nv);
    // two passes keep their partial sums in y: the argmax form without y stays on mma.sync
    if (passes > 1 && !a.y) return false;
    if (a.C % kTcChunk != 0 || pass_blocks(int(a.C / kTcChunk), passes) > tc_build_warps(nv) * kTcMaxJobs) return false;
    if (tc_smem_bytes(a.C, nv) > size_t(227) * 1024) return false;
    if (reinterpret_cast<uintptr_t>(a.w) % 16 != 0 || reinterpret_cast<uintptr_t>(a.x) % 16 != 0) return false;
    // every 64-row unit inside one scale row, every 128-column block inside one scale column block
    if (!chunks_uniform(a.R, a.SR, kTcUnit) || !chunks_uniform(a.C, a.SC, kTcChunk)) return false;
    return encode_tiled() != nullptr;
}

qmv_status launch_tc(const F8Args &a, int batch, bool am, cudaStream_t s, int &blocks_out) {
    CUtensorMap map;
    if (!weight_map(a, map)) return QMV_ERR_CUDA;
    const size_t smem = tc_smem_bytes(a.C, tc_slots(batch));
    const int64_t units = (a.R + kTcUnit - 1) / kTcUnit;
    int64_t blocks = sm_count();
    if (blocks > units) blocks = units;
    if (am && blocks > QMV_ARGMAX_MAX_BLOCKS) blocks = QMV_ARGMAX_MAX_BLOCKS;
    blocks_out = int(blocks);
    if (am) {
        auto kern = f8_tc_kernel<true>;
        if (!allow_smem(reinterpret_cast<const void *>(kern), smem)) return QMV_ERR_CUDA;
        return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(kTcThreads), smem, s, map, a, batch));
    }
    auto kern = f8_tc_kernel<false>;
    if (!allow_smem(reinterpret_cast<const void *>(kern), smem)) return QMV_ERR_CUDA;
    return from_cuda(launch_pdl(kern, dim3(unsigned(blocks)), dim3(kTcThreads), smem, s, map, a, batch));
}

qmv_status tc_wait_timeouts(unsigned long long *count) {
    return from_cuda(cudaMemcpyFromSymbol(count, g_tc_timeouts, sizeof(*count)));
}

}  // namespace f8

qmv_status f8_tc_wait_timeouts(unsigned long long *count) { return f8::tc_wait_timeouts(count); }

}  // namespace qmv
