// cq_kernels.cu -- CQ kernels for sm_103a: activation preparation, dense row
// gather and the packed-row matvec.
//
// Method: needle.js tutorial "Inference engine, part 2: kernels and token
// step" -- section 1 (unnormalised FWHT, strides 1, 2, 4, ... ascending),
// section 2 (prepare: pad, per-group FWHT, times 1/sqrt(group)), section 3
// (y[r] = sum_g norm[r,g] * sum_k codebook[index(r,k)] * prepared[k], and the
// 2-bit byte lookup table), "Row gather" (levels times norm, normalised FWHT,
// unpadded columns).  Matrix layout: "part 1: loader and tokenizer",
// section 4 (CqMatrix).
//
// Bit-exactness of prepare and row gather: every butterfly is a single
// float32 add or subtract (__fadd_rn/__fsub_rn, never contracted), stages run
// in ascending stride order, and the 1/sqrt(G) scale is a float64 product
// rounded once to float32 -- the float32-staged semantics of the page's
// Float32Array code.  Within one stage the butterflies are independent, so
// spreading them over lanes changes no result.
#include <cuda_fp16.h>
#include <stdint.h>

#include "fwht_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// Column k's index in a packed row: bits [k*bits, k*bits+bits) of the row's
// little-endian bit stream.  Reads the second byte only when the code
// straddles a byte boundary (that byte then lies inside the row).
__device__ __forceinline__ int cq_index(const uint8_t *row, int64_t k, int bits) {
    int64_t t = k * bits;
    int64_t byte = t >> 3;
    int sh = int(t & 7);
    unsigned v = __ldg(row + byte);
    if (sh + bits > 8) v |= unsigned(__ldg(row + byte + 1)) << 8;
    return int((v >> sh) & ((1u << bits) - 1u));
}

// ---------------------------------------------------------------------------
// prepare and row gather: one "group job" = one (vector or row id, group)
// ---------------------------------------------------------------------------

enum class GMode { Prepare, Gather };

struct GroupArgs {
    int64_t input, P, G, nG;
    int64_t njobs;  // vectors (prepare) or ids (gather)
    Scale s;        // RN64(1/sqrt(G)), and its float32 split
    float *out;
    // prepare
    const float *x;
    // gather
    const uint8_t *packed;
    const uint16_t *norms;
    const float *codebook;
    int64_t row_bytes, output;
    int bits;
    const int32_t *rows;
    int32_t *status;
};

// Per-thread copy of the codebook for the gather: lane l holds level l
// (2^bits <= 32), so a level is one warp shuffle away once the index is known.
template <GMode M>
__device__ __forceinline__ float codebook_lane(const GroupArgs &a, int lane) {
    if (M == GMode::Prepare) return 0.0f;
    return lane < (1 << a.bits) ? __ldg(a.codebook + lane) : 0.0f;
}

// The value entering the transform at column `col` of job `j` (`valid`
// false: a padding lane of a partial warp, value 0), and whether the job's
// row id is out of range (gather only).  Every lane of the warp must call it
// together: the gather's level lookup is a warp shuffle.
template <GMode M>
__device__ __forceinline__ float group_load(const GroupArgs &a, int64_t j, int64_t col, bool valid,
                                            float cb_lane, bool &bad) {
    if (M == GMode::Prepare) {
        bad = false;
        return (valid && col < a.input) ? __ldg(a.x + j * a.input + col) : 0.0f;
    } else {
        int idx = 0;
        float n = 0.0f;
        bad = false;
        if (valid) {
            const int64_t r = __ldg(a.rows + j);
            bad = (r < 0 || r >= a.output);
            if (!bad) {
                n = half_bits_to_float(__ldg(a.norms + r * a.nG + col / a.G));
                idx = cq_index(a.packed + r * a.row_bytes, col, a.bits);
            }
        }
        const float level = __shfl_sync(kFull, cb_lane, idx);
        return (valid && !bad) ? __fmul_rn(level, n) : 0.0f;
    }
}

template <GMode M>
__device__ __forceinline__ void group_store(const GroupArgs &a, int64_t j, int64_t col, float v,
                                           bool bad) {
    if (M == GMode::Prepare) {
        a.out[j * a.P + col] = v;
    } else {
        if (col < a.input) a.out[j * a.input + col] = bad ? 0.0f : v;
        if (bad && a.status) *a.status = int32_t(QMV_ERR_ROW_ID);
    }
}

// G <= 32: each warp covers 32 consecutive elements of the [njobs, P] space
// (groups never straddle a warp since G divides 32 and P).
template <GMode M>
__global__ void __launch_bounds__(256) group_small_kernel(GroupArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t flat = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x);
    const int64_t total = a.njobs * a.P;
    const bool valid = flat < total;
    const int64_t j = valid ? flat / a.P : 0;
    const int64_t col = valid ? flat - j * a.P : 0;
    bool bad = false;
    float v[1];
    v[0] = group_load<M>(a, j, col, valid, codebook_lane<M>(a, lane), bad);
    fwht_warp<1>(v, int(a.G), lane);
    scale_rn_all<1>(v, a.s);
    if (valid) group_store<M>(a, j, col, v[0], bad);
}

// 64 <= G <= 1024: one warp per group job, E = G/32 elements per lane.
template <GMode M, int E>
__global__ void __launch_bounds__(256) group_warp_kernel(GroupArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (job >= a.njobs * a.nG) return;  // whole warp leaves together
    const int64_t j = job / a.nG, g = job - j * a.nG;
    const int64_t col0 = g * a.G + int64_t(lane) * E;
    const float cbl = codebook_lane<M>(a, lane);
    float v[E];
    bool bad = false;
#pragma unroll
    for (int e = 0; e < E; e++) v[e] = group_load<M>(a, j, col0 + e, true, cbl, bad);
    fwht_warp<E>(v, int(a.G), lane);
    scale_rn_all<E>(v, a.s);
#pragma unroll
    for (int e = 0; e < E; e++) group_store<M>(a, j, col0 + e, v[e], bad);
}

// G > 1024: one block per group job, the group staged in shared memory and
// one stage per barrier.
template <GMode M>
__global__ void __launch_bounds__(1024) group_block_kernel(GroupArgs a) {
    extern __shared__ float sm[];
    pdl_wait();
    pdl_trigger();
    const int64_t job = blockIdx.x;
    const int64_t j = job / a.nG, g = job - j * a.nG;
    const int G = int(a.G);
    const float cbl = codebook_lane<M>(a, threadIdx.x & 31);
    bool bad = false;
    // G is a multiple of blockDim, so every lane runs the same iterations
    for (int i = threadIdx.x; i < G; i += blockDim.x)
        sm[i] = group_load<M>(a, j, g * a.G + i, true, cbl, bad);
    for (int h = 1; h < G; h <<= 1) {
        __syncthreads();
        for (int t = threadIdx.x; t < G / 2; t += blockDim.x) {
            int i = ((t & ~(h - 1)) << 1) | (t & (h - 1));
            float x0 = sm[i], x1 = sm[i + h];
            sm[i] = __fadd_rn(x0, x1);
            sm[i + h] = __fsub_rn(x0, x1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G; i += blockDim.x)
        group_store<M>(a, j, g * a.G + i, scale_rn(sm[i], a.s), bad);
}

template <GMode M>
qmv_status launch_group(const GroupArgs &a, cudaStream_t s) {
    const int64_t jobs = a.njobs * a.nG;
    const int64_t kMaxGrid = 2147483647;
    if ((a.G <= 32 && (a.njobs * a.P + 255) / 256 > kMaxGrid) ||
        (a.G > 32 && a.G <= 1024 && (jobs * 32 + 255) / 256 > kMaxGrid) || jobs > kMaxGrid)
        return QMV_ERR_OVERFLOW;
    cudaError_t e = cudaSuccess;
    if (a.G <= 32) {
        int64_t threads = a.njobs * a.P;
        int64_t blocks = (threads + 255) / 256;
        e = launch_pdl(group_small_kernel<M>, dim3(unsigned(blocks)), dim3(256), 0, s, a);
    } else if (a.G <= 1024) {
        int64_t blocks = (jobs * 32 + 255) / 256;
        const dim3 grid{unsigned(blocks)};
        switch (a.G) {
            case 64: e = launch_pdl(group_warp_kernel<M, 2>, grid, dim3(256), 0, s, a); break;
            case 128: e = launch_pdl(group_warp_kernel<M, 4>, grid, dim3(256), 0, s, a); break;
            case 256: e = launch_pdl(group_warp_kernel<M, 8>, grid, dim3(256), 0, s, a); break;
            case 512: e = launch_pdl(group_warp_kernel<M, 16>, grid, dim3(256), 0, s, a); break;
            default: e = launch_pdl(group_warp_kernel<M, 32>, grid, dim3(256), 0, s, a); break;
        }
    } else {
        size_t smem = size_t(a.G) * sizeof(float);
        if (!allow_smem(reinterpret_cast<const void *>(group_block_kernel<M>), smem)) return QMV_ERR_CUDA;
        e = launch_pdl(group_block_kernel<M>, dim3(unsigned(jobs)), dim3(1024), smem, s, a);
    }
    return from_cuda(e);
}

GroupArgs group_args(const qmv_cq_matrix &m) {
    GroupArgs a = {};
    a.input = m.input;
    a.P = m.input_padded;
    a.G = m.group;
    a.nG = m.input_padded / m.group;
    a.s = make_scale(1.0 / sqrt(double(m.group)));
    a.packed = m.packed;
    a.norms = m.norms;
    a.codebook = m.codebook;
    a.row_bytes = m.row_bytes;
    a.output = m.output;
    a.bits = m.bits;
    return a;
}

// ---------------------------------------------------------------------------
// Matrix sets.  cq_matvec (one matrix), cq_matvec_multi and cq_prepare_matvec
// (several matrices sharing input width, group, bits and codebook -- needle-2
// section 6: one prepared activation serves phiPre, phiPost and phiResidual;
// section 7: Q, K and V of one input) run the same kernels.  The units of all
// matrices (rows, or groups of RPW rows for the table kernel) form one space;
// unit u belongs to matrix i when first[i] <= u < first[i+1].  With FUSED the
// activation is prepared inside every block (same butterflies and rounding as
// cq_prepare, so the results are bitwise those of cq_prepare + cq_matvec).
// ---------------------------------------------------------------------------

struct CqSet {
    int nmats, bits;
    int64_t input, P, G, nG, row_bytes;
    const float *codebook;
    int64_t output[QMV_MAX_MATRICES];
    const uint8_t *packed[QMV_MAX_MATRICES];
    const uint16_t *norms[QMV_MAX_MATRICES];
    float *y[QMV_MAX_MATRICES];
    int64_t first[QMV_MAX_MATRICES + 1];
    const float *p;        // prepared activation [B, P] (not FUSED)
    const float *x;        // raw activation [B, input] (FUSED)
    float *prepared_out;   // FUSED: block 0 also stores the prepared vector (may be NULL)
    Scale s;               // RN64(1/sqrt(G)), and its float32 split
};

// Matrix of unit u, scanning on from matrix i (units of a warp only grow).
__device__ __forceinline__ int set_matrix(const CqSet &c, int64_t u, int i) {
    while (i + 1 < c.nmats && u >= c.first[i + 1]) i++;
    return i;
}

// ---- in-block prepare (FUSED): x -> sp[B][P] in shared memory -------------
template <int E>
__device__ __forceinline__ void prep_warp_jobs(const CqSet &c, int B, float *sp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const bool store = c.prepared_out && blockIdx.x == 0;
    const int64_t jobs = int64_t(B) * c.nG;
    for (int64_t job = warp; job < jobs; job += nw) {
        const int64_t v = job / c.nG, g = job - v * c.nG;
        const int64_t col0 = g * c.G + int64_t(lane) * E;
        float val[E];
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int64_t col = col0 + e;
            val[e] = col < c.input ? __ldg(c.x + v * c.input + col) : 0.0f;
        }
        fwht_warp<E>(val, int(c.G), lane);
        scale_rn_all<E>(val, c.s);
#pragma unroll
        for (int e = 0; e < E; e++) {
            const float o = val[e];
            sp[v * c.P + col0 + e] = o;
            if (store) c.prepared_out[v * c.P + col0 + e] = o;
        }
    }
}

// G <= 32: each warp transforms 32 consecutive elements of the [B, P] space.
__device__ __forceinline__ void prep_small(const CqSet &c, int B, float *sp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const bool store = c.prepared_out && blockIdx.x == 0;
    const int64_t total = int64_t(B) * c.P;
    for (int64_t chunk = warp; chunk * 32 < total; chunk += nw) {
        const int64_t flat = chunk * 32 + lane;
        const bool valid = flat < total;
        const int64_t v = valid ? flat / c.P : 0, col = valid ? flat - v * c.P : 0;
        float val[1];
        val[0] = (valid && col < c.input) ? __ldg(c.x + v * c.input + col) : 0.0f;
        fwht_warp<1>(val, int(c.G), lane);
        scale_rn_all<1>(val, c.s);
        if (valid) {
            const float o = val[0];
            sp[flat] = o;
            if (store) c.prepared_out[flat] = o;
        }
    }
}

__device__ __forceinline__ void block_prepare(const CqSet &c, int B, float *sp) {
    switch (c.G) {
        case 64: prep_warp_jobs<2>(c, B, sp); break;
        case 128: prep_warp_jobs<4>(c, B, sp); break;
        case 256: prep_warp_jobs<8>(c, B, sp); break;
        case 512: prep_warp_jobs<16>(c, B, sp); break;
        case 1024: prep_warp_jobs<32>(c, B, sp); break;
        default: prep_small(c, B, sp); break;  // G <= 32 (fused launches never take G > 1024)
    }
}

// ---------------------------------------------------------------------------
// General kernel: any bits, group, width, batch and alignment.  One warp per
// row; lane l takes columns l, l+32, ...; each element contributes
// (codebook level * norm) * prepared in a float32 FMA, then a fixed-order
// warp reduction.
// ---------------------------------------------------------------------------
template <int B, bool FUSED>
__global__ void __launch_bounds__(256) cq_matvec_general_kernel(CqSet c) {
    __shared__ float cb[32];
    extern __shared__ __align__(16) float sp_dyn[];
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < (1 << c.bits)) cb[threadIdx.x] = c.codebook[threadIdx.x];
    const float *p = c.p;
    if (FUSED) {
        block_prepare(c, B, sp_dyn);
        p = sp_dyn;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t P = c.P, nG = c.nG;
    const int lg = __ffsll(c.G) - 1;
    int mi = 0;
    for (int64_t u = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; u < c.first[c.nmats];
         u += nwarps) {
        mi = set_matrix(c, u, mi);
        const int64_t r = u - c.first[mi];
        const uint8_t *row = c.packed[mi] + r * c.row_bytes;
        const uint16_t *nrow = c.norms[mi] + r * nG;
        float acc[B];
#pragma unroll
        for (int v = 0; v < B; v++) acc[v] = 0.0f;
        for (int64_t k = lane; k < P; k += 32) {
            const float n = half_bits_to_float(__ldg(nrow + (k >> lg)));
            const float wv = cb[cq_index(row, k, c.bits)] * n;
#pragma unroll
            for (int v = 0; v < B; v++) acc[v] = fmaf(wv, FUSED ? p[v * P + k] : __ldg(p + v * P + k), acc[v]);
        }
#pragma unroll
        for (int v = 0; v < B; v++) {
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) acc[v] += __shfl_xor_sync(kFull, acc[v], d);
        }
        if (lane == 0) {
            const int64_t out = c.output[mi];
#pragma unroll
            for (int v = 0; v < B; v++) c.y[mi][v * out + r] = acc[v];
        }
    }
}

// ---------------------------------------------------------------------------
// 2-bit / batch-1 kernel with the activation folded into a nibble table.  The
// page's 2-bit loop looks up four levels per byte (section 3); here each
// table entry already holds the two products of one nibble:
//   T[nib][c2] = codebook[nib & 3] * p[2*c2] + codebook[nib >> 2] * p[2*c2+1]
// so every 4-bit code pair costs one shared-memory load and half a packed
// add (add.f32x2 sums two lookups at once).
//
// Lanes.  A row of P columns is CPR = P/64 chunks of 16 bytes (64 codes).
// Lane l of a warp owns chunk q = l % CPR of row rho = l / CPR (RPW = 32/CPR
// rows per warp, one "unit") and walks its 32 nibbles in the order rho,
// rho+1, ... (its 16 bytes rotated right by 4*rho bits).
//
// Table layout (bytes): page q at 4096 q, nibble row nib at 256 nib inside
// it, slot s (0..63) at 4 s; chunk q's column pair j is stored at slots
// (j + RPW q) % 32 and that + 32.  At step t lane (rho, q) reads slot
// t + rho + RPW q, so the 32 lanes of a warp always hit 32 distinct banks,
// and its address is one byte permute of the nibble (byte 1, with q's low
// bits pre-set in the high half of the byte) and a per-lane word (slot base
// in byte 0, q's high bit in byte 2), plus the immediate 4 t.
//
// Work split.  One block of 512 threads per SM (kCq2Threads, <= 64
// registers), so a second call's block fits beside it; the units are split
// evenly over the blocks and, inside a block, warp w takes units w, w + 16,
// ....  The first kCq2Pre units of every warp are loaded into registers
// before the dependency wait -- while the preceding call is still running --
// and the block lets its dependents launch at once (on grids of at most half
// the SMs, only after the wait).  After the wait: the
// prepared vector and codebook, the table build, the lookups.
//
// Shared memory: 64*P bytes (4 KB per chunk) plus 4*P for the prepared vector
// when FUSED.  Requirements (checked by the launcher): bits == 2, batch == 1,
// P in {256, 512, 1024, 2048}, group >= 64, 16-byte aligned packed rows.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void cq2_load(uint4 &d, float &n, const CqSet &c, int mi, int64_t r, int q, int g) {
    d = make_uint4(0, 0, 0, 0);
    n = 0.0f;
    if (r < c.output[mi]) {
        const uint4 *src = reinterpret_cast<const uint4 *>(c.packed[mi] + r * c.row_bytes) + q;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
                     : "l"(src));
        n = half_bits_to_float(__ldg(c.norms[mi] + r * c.nG + g));
    }
}

constexpr int kCq2Threads = 512;
constexpr int kCq2Warps = kCq2Threads / 32;
constexpr int kCq2Pre = 4;  // units per warp loaded before the dependency wait

template <int CPR, bool FUSED>
__global__ void __launch_bounds__(kCq2Threads, FUSED ? 1 : 2) cq2_table_kernel(CqSet c, int64_t upb, int late_trigger) {
    constexpr int RPW = 32 / CPR;
    constexpr int P = CPR * 64;
    extern __shared__ __align__(16) unsigned char table_raw[];
    float *table = reinterpret_cast<float *>(table_raw);
    float *sp = reinterpret_cast<float *>(table_raw + 64 * P);  // FUSED: prepared vector

    if (!late_trigger) pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rho = lane / CPR, q = lane % CPR;
    const int g = (q * 64) / int(c.G);
    const int64_t nunits = c.first[c.nmats];
    const int64_t ub0 = int64_t(blockIdx.x) * upb;
    const int64_t ub1 = min(nunits, ub0 + upb);

    // this warp's first units, into registers while the preceding call runs
    uint4 d[kCq2Pre];
    float n[kCq2Pre];
    int mis[kCq2Pre];
    {
        int mi = set_matrix(c, ub0, 0);
#pragma unroll
        for (int k = 0; k < kCq2Pre; k++) {
            const int64_t u = ub0 + warp + int64_t(k) * kCq2Warps;
            d[k] = make_uint4(0, 0, 0, 0);
            n[k] = 0.0f;
            mis[k] = mi;
            if (u < ub1) {
                mi = set_matrix(c, u, mi);
                mis[k] = mi;
                cq2_load(d[k], n[k], c, mi, (u - c.first[mi]) * RPW + rho, q, g);
            }
        }
    }
    pdl_wait();
    if (late_trigger) pdl_trigger();

    const float *pv = c.p;
    if (FUSED) {
        block_prepare(c, 1, sp);
        __syncthreads();
        pv = sp;
    }
    // ---- build the table: a job is one column pair and half of its 16
    // entries; consecutive lanes take consecutive pairs, so every store of a
    // warp hits 32 distinct banks ----
    {
        float cbv[4];
#pragma unroll
        for (int i = 0; i < 4; i++) cbv[i] = __ldg(c.codebook + i);
        constexpr int NPAIR = CPR * 32;
        for (int job = threadIdx.x; job < 2 * NPAIR; job += blockDim.x) {
            const int pair = job % NPAIR, half = job / NPAIR;
            const int qq = pair >> 5, j = pair & 31;
            const int col = qq * 64 + 2 * j;
            const float p0 = FUSED ? pv[col] : __ldg(pv + col);
            const float p1 = FUSED ? pv[col + 1] : __ldg(pv + col + 1);
            float lo_prod[4];
#pragma unroll
            for (int i = 0; i < 4; i++) lo_prod[i] = cbv[i] * p0;
            float *blk = table + qq * 1024 + ((j + RPW * qq) & 31);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int hi = 2 * half + h;
                const float chi = half ? cbv[2 + h] : cbv[h];
#pragma unroll
                for (int lo = 0; lo < 4; lo++) {
                    const float v = fmaf(chi, p1, lo_prod[lo]);
                    float *e = blk + (lo | (hi << 2)) * 64;
                    e[0] = v;
                    e[32] = v;
                }
            }
        }
    }
    __syncthreads();

    const unsigned q4 = (unsigned(q & 15) << 4) * 0x01010101u;
    const unsigned lane_word = unsigned(4 * (rho + RPW * q)) | (unsigned(q >> 4) << 16);
    const char *tb = reinterpret_cast<const char *>(table);
    const unsigned sh = 4u * unsigned(rho);
    auto unit = [&](const uint4 &dd, float nv, int mi, int64_t u) {
        // rotate the 128-bit chunk right by 4*rho bits; every word then gives
        // its even nibbles (one per byte) and its odd nibbles
        unsigned w[4];
        w[0] = __funnelshift_r(dd.x, dd.y, sh);
        w[1] = __funnelshift_r(dd.y, dd.z, sh);
        w[2] = __funnelshift_r(dd.z, dd.w, sh);
        w[3] = __funnelshift_r(dd.w, dd.x, sh);
        float2 s2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const unsigned ev = (w[i] & 0x0f0f0f0fu) | q4, od = ((w[i] >> 4) & 0x0f0f0f0fu) | q4;
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
                const int t = 8 * i + 2 * kk;
                const unsigned ae = __byte_perm(ev, lane_word, 0x7604u | (unsigned(kk) << 4));
                const unsigned ao = __byte_perm(od, lane_word, 0x7604u | (unsigned(kk) << 4));
                const float te = *reinterpret_cast<const float *>(tb + ae + 4 * t);
                const float to = *reinterpret_cast<const float *>(tb + ao + 4 * (t + 1));
                s2 = __fadd2_rn(s2, make_float2(te, to));
            }
        }
        float acc = nv * (s2.x + s2.y);
#pragma unroll
        for (int dd2 = CPR / 2; dd2 >= 1; dd2 >>= 1) acc += __shfl_xor_sync(kFull, acc, dd2);
        const int64_t r = (u - c.first[mi]) * RPW + rho;
        if (q == 0 && r < c.output[mi]) c.y[mi][r] = acc;
    };
#pragma unroll
    for (int k = 0; k < kCq2Pre; k++) {
        const int64_t u = ub0 + warp + int64_t(k) * kCq2Warps;
        if (u < ub1) unit(d[k], n[k], mis[k], u);  // warp-uniform
    }
    // larger matrices: the remaining units, kCq2Pre at a time
    for (int64_t base = ub0 + warp + int64_t(kCq2Pre) * kCq2Warps; base < ub1;
         base += int64_t(kCq2Pre) * kCq2Warps) {
        int mi = mis[kCq2Pre - 1];
#pragma unroll
        for (int k = 0; k < kCq2Pre; k++) {
            const int64_t u = base + int64_t(k) * kCq2Warps;
            d[k] = make_uint4(0, 0, 0, 0);
            n[k] = 0.0f;
            mis[k] = mi;
            if (u < ub1) {
                mi = set_matrix(c, u, mi);
                mis[k] = mi;
                cq2_load(d[k], n[k], c, mi, (u - c.first[mi]) * RPW + rho, q, g);
            }
        }
#pragma unroll
        for (int k = 0; k < kCq2Pre; k++) {
            const int64_t u = base + int64_t(k) * kCq2Warps;
            if (u < ub1) unit(d[k], n[k], mis[k], u);
        }
    }
}

template <int CPR, bool FUSED>
qmv_status launch_cq2_table(CqSet c, cudaStream_t s) {
    constexpr int RPW = 32 / CPR;
    const size_t smem = size_t(64) * CPR * 64 + (FUSED ? size_t(4) * CPR * 64 : 0);
    const void *kp = reinterpret_cast<const void *>(cq2_table_kernel<CPR, FUSED>);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    c.first[0] = 0;
    for (int i = 0; i < c.nmats; i++) c.first[i + 1] = c.first[i] + (c.output[i] + RPW - 1) / RPW;
    const int64_t nunits = c.first[c.nmats];
    // one block per SM at most (leaving room for the next call's block), and
    // no more blocks than a warp's worth of units each
    int64_t blocks = (nunits + kCq2Warps - 1) / kCq2Warps;
    if (blocks > sm_count()) blocks = sm_count();
    if (blocks < 1) blocks = 1;
    const int64_t upb = (nunits + blocks - 1) / blocks;
    // Dependents launch at entry, except on grids of at most half the SMs,
    // where they are let in after the wait: 2048 x 512 ran 1.57 against 1.70
    // us per call in chains, while 32768 x 512 ran 3.30 against 2.96.
    const int late = 2 * blocks <= sm_count() ? 1 : 0;
    return from_cuda(launch_pdl(cq2_table_kernel<CPR, FUSED>, dim3(unsigned(blocks)), dim3(kCq2Threads), smem, s, c, upb, late));
}

template <int B, bool FUSED>
qmv_status launch_cq_general(CqSet c, cudaStream_t s) {
    const size_t smem = FUSED ? size_t(4) * B * c.P : 0;
    const void *kp = reinterpret_cast<const void *>(cq_matvec_general_kernel<B, FUSED>);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    c.first[0] = 0;
    for (int i = 0; i < c.nmats; i++) c.first[i + 1] = c.first[i] + c.output[i];
    const int blocks = grid_blocks(kp, 256, smem, c.first[c.nmats]);
    return from_cuda(launch_pdl(cq_matvec_general_kernel<B, FUSED>, dim3(unsigned(blocks)), dim3(256), smem, s, c));
}

// ---------------------------------------------------------------------------
// Vectorised kernel: any bits (2..5), batch 1..8, group >= 16, P % 16 == 0,
// 2-byte aligned packed rows (row_bytes = 2 * bits * P / 16 is even).
//
// Lane l takes 16-column chunks ch = l, l+32, ... of a row (one warp per
// row): the chunk's 16 codes are 2 * bits bytes, read as `bits` 16-bit words
// into one 80-bit field, and code e is bits [bits*e, bits*e + bits) of it.  The
// level is a warp shuffle from the lane that holds it (lane i keeps codebook
// level i); the chunk lies inside one group, so the group's norm multiplies
// the chunk's partial sum once.  The prepared vectors are staged in shared
// memory with a 17-word pitch per chunk, so at every step the 32 lanes read
// 32 distinct banks.
// ---------------------------------------------------------------------------

// Code e (compile-time) of a 16-code chunk held as lo (bits 0..63) and hi
// (bits 64..79).
template <int BITS, int E>
__device__ __forceinline__ int chunk_code(uint64_t lo, uint32_t hi) {
    constexpr int S = BITS * E;
    constexpr unsigned M = (1u << BITS) - 1u;
    if constexpr (S + BITS <= 64) {
        return int(unsigned(lo >> S) & M);
    } else if constexpr (S >= 64) {
        return int((hi >> (S - 64)) & M);
    } else {
        return int((unsigned(lo >> S) | (hi << (64 - S))) & M);
    }
}

template <int BITS, int B, bool FUSED>
__global__ void __launch_bounds__(256) cq_vec_kernel(CqSet c) {
    // [B][P] prepared vectors when FUSED (as the in-block prepare writes
    // them), then [B][P/16][17] padded
    extern __shared__ __align__(16) float vec_smem[];
    float *spad = vec_smem + (FUSED ? int64_t(B) * c.P : 0);
    const int lane = threadIdx.x & 31;
    const int64_t P = c.P;
    const int nch = int(P >> 4);
    const int lg = __ffsll(c.G) - 1;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int steps = (nch + 31) >> 5;
    const int64_t nunits = c.first[c.nmats];
    // chunk ch of row r of matrix mi: its 16 codes and its group's norm
    auto load_chunk = [&](int mi, int64_t r, int ch, uint64_t &lo, uint32_t &hi, float &n) {
        lo = 0;
        hi = 0;
        n = 0.0f;
        if (ch < nch) {
            const uint16_t *src = reinterpret_cast<const uint16_t *>(c.packed[mi] + r * c.row_bytes) + ch * BITS;
#pragma unroll
            for (int i = 0; i < BITS; i++) {
                const uint64_t h = __ldg(src + i);
                if (i < 4)
                    lo |= h << (16 * i);
                else
                    hi = uint32_t(h);
            }
            n = half_bits_to_float(__ldg(c.norms[mi] + r * c.nG + ((int64_t(ch) << 4) >> lg)));
        }
    };
    // this warp's first row, first chunk step, and the codebook: loaded
    // before the dependency wait (the matrices are read-only model data).
    // Dependents are let in only after the wait: triggered at entry, chains
    // of these short calls ran slower (3-5-bit 2048 x 512: 3.5 against 2.1 us).
    int64_t u = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    int mi = 0;
    uint64_t lo0 = 0;
    uint32_t hi0 = 0;
    float n0 = 0.0f;
    if (u < nunits) {
        mi = set_matrix(c, u, 0);
        load_chunk(mi, u - c.first[mi], lane, lo0, hi0, n0);
    }
    const float cb_lane = lane < (1 << BITS) ? __ldg(c.codebook + lane) : 0.0f;
    pdl_wait();
    pdl_trigger();
    const float *psrc = c.p;
    if (FUSED) {
        block_prepare(c, B, vec_smem);
        __syncthreads();
        psrc = vec_smem;
    }
    for (int64_t i = threadIdx.x; i < int64_t(B) * P; i += blockDim.x) {
        const int64_t v = i / P, k = i - v * P;
        spad[(v * nch + (k >> 4)) * 17 + (k & 15)] = FUSED ? psrc[i] : __ldg(psrc + i);
    }
    __syncthreads();
    bool first = true;
    for (; u < nunits; u += nwarps) {
        mi = set_matrix(c, u, mi);
        const int64_t r = u - c.first[mi];
        float acc[B];
#pragma unroll
        for (int v = 0; v < B; v++) acc[v] = 0.0f;
        for (int j = 0; j < steps; j++) {  // warp-uniform trip count: every lane shuffles
            const int ch = lane + 32 * j;
            const bool valid = ch < nch;
            uint64_t lo;
            uint32_t hi;
            float n;
            if (first && j == 0) {
                lo = lo0;
                hi = hi0;
                n = n0;
            } else {
                load_chunk(mi, r, ch, lo, hi, n);
            }
            const float *pp = spad + (valid ? ch : 0) * 17;
            float part[B];
#pragma unroll
            for (int v = 0; v < B; v++) part[v] = 0.0f;
#define QMV_CQ_VEC_STEP(E)                                                                   \
    {                                                                                        \
        const float lv = __shfl_sync(kFull, cb_lane, chunk_code<BITS, E>(lo, hi));           \
        _Pragma("unroll") for (int v = 0; v < B; v++) part[v] =                               \
            fmaf(lv, pp[v * nch * 17 + E], part[v]);                                         \
    }
            QMV_CQ_VEC_STEP(0) QMV_CQ_VEC_STEP(1) QMV_CQ_VEC_STEP(2) QMV_CQ_VEC_STEP(3)
            QMV_CQ_VEC_STEP(4) QMV_CQ_VEC_STEP(5) QMV_CQ_VEC_STEP(6) QMV_CQ_VEC_STEP(7)
            QMV_CQ_VEC_STEP(8) QMV_CQ_VEC_STEP(9) QMV_CQ_VEC_STEP(10) QMV_CQ_VEC_STEP(11)
            QMV_CQ_VEC_STEP(12) QMV_CQ_VEC_STEP(13) QMV_CQ_VEC_STEP(14) QMV_CQ_VEC_STEP(15)
#undef QMV_CQ_VEC_STEP
            if (valid) {  // (a lane past the row's end shuffled with the others, adds nothing)
#pragma unroll
                for (int v = 0; v < B; v++) acc[v] = fmaf(part[v], n, acc[v]);
            }
        }
        first = false;
#pragma unroll
        for (int v = 0; v < B; v++) {
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) acc[v] += __shfl_xor_sync(kFull, acc[v], d);
        }
        if (lane == 0) {
            const int64_t out = c.output[mi];
#pragma unroll
            for (int v = 0; v < B; v++) c.y[mi][v * out + r] = acc[v];
        }
    }
}

template <int BITS, int B, bool FUSED>
qmv_status launch_cq_vec(CqSet c, cudaStream_t s) {
    const size_t smem = size_t(4) * B * (c.P / 16) * 17 + (FUSED ? size_t(4) * B * c.P : 0);
    const void *kp = reinterpret_cast<const void *>(cq_vec_kernel<BITS, B, FUSED>);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    c.first[0] = 0;
    for (int i = 0; i < c.nmats; i++) c.first[i + 1] = c.first[i] + c.output[i];
    const int blocks = grid_blocks(kp, 256, smem, c.first[c.nmats]);
    return from_cuda(launch_pdl(cq_vec_kernel<BITS, B, FUSED>, dim3(unsigned(blocks)), dim3(256), smem, s, c));
}

template <int BITS, bool FUSED>
qmv_status launch_cq_vec_b(const CqSet &c, int batch, cudaStream_t s) {
    switch (batch) {
        case 1: return launch_cq_vec<BITS, 1, FUSED>(c, s);
        case 2: return launch_cq_vec<BITS, 2, FUSED>(c, s);
        case 3: return launch_cq_vec<BITS, 3, FUSED>(c, s);
        case 4: return launch_cq_vec<BITS, 4, FUSED>(c, s);
        case 5: return launch_cq_vec<BITS, 5, FUSED>(c, s);
        case 6: return launch_cq_vec<BITS, 6, FUSED>(c, s);
        case 7: return launch_cq_vec<BITS, 7, FUSED>(c, s);
        default: return launch_cq_vec<BITS, 8, FUSED>(c, s);
    }
}

template <bool FUSED>
qmv_status launch_set(const CqSet &c, int batch, bool all_aligned16, bool all_aligned2, cudaStream_t s) {
    const int64_t P = c.P;
    // The kernel depends on the matrices' common shape only (never on their
    // row counts or on FUSED), so a set call, its per-matrix calls and the
    // fused prepare all run the same arithmetic.  (At 2048 rows the
    // vectorised kernel would be 0.2 us faster than the table; at 32768 rows
    // it is 2.3x slower.)
    const bool table_ok = c.bits == 2 && batch == 1 && c.G >= 64 &&
                          (P == 256 || P == 512 || P == 1024 || P == 2048) && all_aligned16;
    if (table_ok) {
        switch (P) {
            case 256: return launch_cq2_table<4, FUSED>(c, s);
            case 512: return launch_cq2_table<8, FUSED>(c, s);
            case 1024: return launch_cq2_table<16, FUSED>(c, s);
            default: return launch_cq2_table<32, FUSED>(c, s);
        }
    }
    // vectorised kernel: group >= 16, P % 16 == 0, 2-byte aligned rows, and the
    // prepared vectors (padded) in shared memory.  The fused variant takes
    // exactly the same cases (it prepares wherever cq_fused_fits holds, so
    // P * batch * 4 <= 96 KB), which keeps cq_prepare_matvec bitwise equal to
    // cq_prepare + cq_matvec.
    if (c.G >= 16 && P % 16 == 0 && all_aligned2 && size_t(4) * batch * (P / 16) * 17 <= 102 * 1024) {
        switch (c.bits) {
            case 2: return launch_cq_vec_b<2, FUSED>(c, batch, s);
            case 3: return launch_cq_vec_b<3, FUSED>(c, batch, s);
            case 4: return launch_cq_vec_b<4, FUSED>(c, batch, s);
            default: return launch_cq_vec_b<5, FUSED>(c, batch, s);
        }
    }
    switch (batch) {
        case 1: return launch_cq_general<1, FUSED>(c, s);
        case 2: return launch_cq_general<2, FUSED>(c, s);
        case 3: return launch_cq_general<3, FUSED>(c, s);
        case 4: return launch_cq_general<4, FUSED>(c, s);
        case 5: return launch_cq_general<5, FUSED>(c, s);
        case 6: return launch_cq_general<6, FUSED>(c, s);
        case 7: return launch_cq_general<7, FUSED>(c, s);
        default: return launch_cq_general<8, FUSED>(c, s);
    }
}

}  // namespace

qmv_status launch_cq_prepare(const qmv_cq_matrix &m, const float *x, int batch, float *prepared,
                             cudaStream_t s) {
    GroupArgs a = group_args(m);
    a.njobs = batch;
    a.x = x;
    a.out = prepared;
    return launch_group<GMode::Prepare>(a, s);
}

qmv_status launch_cq_dequantize_row(const qmv_cq_matrix &m, const int32_t *rows, int64_t n, float *out,
                                    int32_t *dev_status, cudaStream_t s) {
    GroupArgs a = group_args(m);
    a.njobs = n;
    a.rows = rows;
    a.status = dev_status;
    a.out = out;
    return launch_group<GMode::Gather>(a, s);
}

bool cq_fused_fits(const qmv_cq_matrix &m, int batch) {
    return m.group <= 1024 && int64_t(batch) * m.input_padded * 4 <= 96 * 1024;
}

qmv_status launch_cq_set(const qmv_cq_matrix *mats, int nmats, const float *p, const float *x,
                         float *prepared_out, int batch, float *const *ys, cudaStream_t s) {
    CqSet c = {};
    const qmv_cq_matrix &m0 = mats[0];
    c.nmats = nmats;
    c.bits = m0.bits;
    c.input = m0.input;
    c.P = m0.input_padded;
    c.G = m0.group;
    c.nG = m0.input_padded / m0.group;
    c.row_bytes = m0.row_bytes;
    c.codebook = m0.codebook;
    c.s = make_scale(1.0 / sqrt(double(m0.group)));
    c.p = p;
    c.x = x;
    c.prepared_out = prepared_out;
    bool aligned16 = true, aligned2 = true;
    for (int i = 0; i < nmats; i++) {
        c.output[i] = mats[i].output;
        c.packed[i] = mats[i].packed;
        c.norms[i] = mats[i].norms;
        c.y[i] = ys[i];
        if (reinterpret_cast<uintptr_t>(mats[i].packed) % 16 != 0) aligned16 = false;
        if (reinterpret_cast<uintptr_t>(mats[i].packed) % 2 != 0) aligned2 = false;
    }
    return x ? launch_set<true>(c, batch, aligned16, aligned2, s) : launch_set<false>(c, batch, aligned16, aligned2, s);
}

qmv_status launch_cq_matvec(const qmv_cq_matrix &m, const float *p, int batch, float *y, cudaStream_t s) {
    float *ys[1] = {y};
    return launch_cq_set(&m, 1, p, nullptr, nullptr, batch, ys, s);
}

}  // namespace qmv
