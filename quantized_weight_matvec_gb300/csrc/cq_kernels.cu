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

// RN32(RN64(v * s)): the page multiplies a float32 element by the float64
// 1/sqrt(group) and stores the product into float32.
__device__ __forceinline__ float scale_f64(float v, double s) {
    return __double2float_rn(__dmul_rn(double(v), s));
}

// Unnormalised FWHT of one group spread over a warp.  For G >= 32 each lane
// holds E = G/32 consecutive elements (element i = lane*E + e); for G < 32
// (E == 1) the warp holds 32/G groups, element i = lane % G.  Stride h is
// in-register while h < E, else a shuffle with lane distance h/E; the lane
// owning the lower index keeps a+b, the upper one keeps a-b.
template <int E>
__device__ __forceinline__ void fwht_warp(float (&v)[E], int G, int lane) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int e = 0; e < E; e++) {
            if ((e & h) == 0) {
                float a = v[e], b = v[e + h];
                v[e] = __fadd_rn(a, b);
                v[e + h] = __fsub_rn(a, b);
            }
        }
    }
    for (int d = 1; d * E < G; d <<= 1) {
        bool upper = (lane & d) != 0;
#pragma unroll
        for (int e = 0; e < E; e++) {
            float o = __shfl_xor_sync(kFull, v[e], d);
            v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
        }
    }
}

// ---------------------------------------------------------------------------
// prepare and row gather: one "group job" = one (vector or row id, group)
// ---------------------------------------------------------------------------

enum class GMode { Prepare, Gather };

struct GroupArgs {
    int64_t input, P, G, nG;
    int64_t njobs;  // vectors (prepare) or ids (gather)
    double s;       // RN64(1/sqrt(G))
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
    if (valid) group_store<M>(a, j, col, scale_f64(v[0], a.s), bad);
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
#pragma unroll
    for (int e = 0; e < E; e++) group_store<M>(a, j, col0 + e, scale_f64(v[e], a.s), bad);
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
        group_store<M>(a, j, g * a.G + i, scale_f64(sm[i], a.s), bad);
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
    a.s = 1.0 / sqrt(double(m.group));
    a.packed = m.packed;
    a.norms = m.norms;
    a.codebook = m.codebook;
    a.row_bytes = m.row_bytes;
    a.output = m.output;
    a.bits = m.bits;
    return a;
}

// ---------------------------------------------------------------------------
// cq_matvec, general kernel: any bits, group, width and alignment.  One warp
// per row; lane l takes columns l, l+32, ...; each element contributes
// (codebook level * norm) * prepared in a float32 FMA, then a fixed-order warp
// reduction.
// ---------------------------------------------------------------------------

template <int B>
__global__ void __launch_bounds__(256) cq_matvec_general_kernel(qmv_cq_matrix m, const float *p,
                                                                float *y) {
    __shared__ float cb[32];
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < (1 << m.bits)) cb[threadIdx.x] = m.codebook[threadIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t P = m.input_padded, nG = P / m.group;
    const int lg = __ffsll(m.group) - 1;
    for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < m.output;
         r += nwarps) {
        const uint8_t *row = m.packed + r * m.row_bytes;
        float acc[B];
#pragma unroll
        for (int v = 0; v < B; v++) acc[v] = 0.0f;
        for (int64_t k = lane; k < P; k += 32) {
            float n = half_bits_to_float(__ldg(m.norms + r * nG + (k >> lg)));
            float wv = cb[cq_index(row, k, m.bits)] * n;
#pragma unroll
            for (int v = 0; v < B; v++) acc[v] = fmaf(wv, __ldg(p + v * P + k), acc[v]);
        }
#pragma unroll
        for (int v = 0; v < B; v++) {
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) acc[v] += __shfl_xor_sync(kFull, acc[v], d);
        }
        if (lane == 0) {
#pragma unroll
            for (int v = 0; v < B; v++) y[v * m.output + r] = acc[v];
        }
    }
}

// ---------------------------------------------------------------------------
// cq_matvec, 2-bit / batch-1 kernel with the activation folded into a nibble
// table.  The page's 2-bit loop looks up four levels per byte (section 3);
// here each table entry already holds the two products of one nibble:
//   T[nib][c2] = codebook[nib & 3] * p[2*c2] + codebook[nib >> 2] * p[2*c2+1]
// so every 4-bit code pair costs one shared-memory load and one add.
//
// Layout.  A row of P columns is CPR = P/64 chunks of 16 bytes (64 codes).
// Lane l of a warp owns chunk q = l % CPR of row rho = l / CPR (RPW = 32/CPR
// rows per warp) and walks its 32 nibbles in the order rho, rho+1, ...
// (its 16 bytes rotated right by 4*rho bits).  Chunk q's entries are stored
// with a bank skew of RPW*q and twice (slots s and s+32), so at step t lane
// (rho, q) reads slot t + rho + RPW*q: the 32 lanes of a warp always hit 32
// distinct banks and the address is a per-lane constant plus 4*t.
//
// Shared memory: 16 nibbles x CPR chunks x 64 slots x 4 B = 64*P bytes.
// Requirements (checked by the launcher): bits == 2, batch == 1,
// P in {256, 512, 1024, 2048}, group >= 64, 16-byte aligned packed rows.
// ---------------------------------------------------------------------------

template <int CPR>
__device__ __forceinline__ void cq2_load(uint4 &d, float &n, const qmv_cq_matrix &m, int64_t r, int q,
                                         int g, int64_t nG) {
    d = make_uint4(0, 0, 0, 0);
    n = 0.0f;
    if (r < m.output) {
        const uint4 *src = reinterpret_cast<const uint4 *>(m.packed + r * m.row_bytes) + q;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
                     : "l"(src));
        n = half_bits_to_float(__ldg(m.norms + r * nG + g));
    }
}

template <int CPR>
__global__ void __launch_bounds__(1024, 1) cq2_table_kernel(qmv_cq_matrix m, const float *p, float *y) {
    constexpr int RPW = 32 / CPR;
    constexpr int P = CPR * 64;
    constexpr int NIB_STRIDE = 4 * P;  // bytes per nibble block
    constexpr int LG_NIB = (P == 256) ? 10 : (P == 512) ? 11 : (P == 1024) ? 12 : 13;
    static_assert((1 << LG_NIB) == NIB_STRIDE, "nibble stride");
    extern __shared__ __align__(16) unsigned char table_raw[];
    float *table = reinterpret_cast<float *>(table_raw);

    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int rho = lane / CPR, q = lane % CPR;
    const int64_t nG = P / m.group;
    const int g = (q * 64) / int(m.group);
    const int64_t ngroups_rows = (m.output + RPW - 1) / RPW;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    int64_t rg = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;

    // the first rows' loads go out before the table is built
    uint4 d;
    float n;
    cq2_load<CPR>(d, n, m, rg * RPW + rho, q, g, nG);

    // ---- build the table (one pass per block): one thread per column pair
    // (chunk q, pair j) loads p once and writes all 16 nibble entries ----
    {
        float cb[4];
#pragma unroll
        for (int i = 0; i < 4; i++) cb[i] = __ldg(m.codebook + i);
        for (int u = threadIdx.x; u < CPR * 32; u += blockDim.x) {
            const int qq = u >> 5, j = u & 31;
            const int col = qq * 64 + 2 * j;
            const float p0 = __ldg(p + col), p1 = __ldg(p + col + 1);
            float lo_prod[4];
#pragma unroll
            for (int i = 0; i < 4; i++) lo_prod[i] = cb[i] * p0;
            const int slot = (j + RPW * qq) & 31;
            float *blk = table + (qq * 256) / 4 + slot;
#pragma unroll
            for (int hi = 0; hi < 4; hi++) {
#pragma unroll
                for (int lo = 0; lo < 4; lo++) {
                    const float v = fmaf(cb[hi], p1, lo_prod[lo]);
                    float *e = blk + (lo | (hi << 2)) * (NIB_STRIDE / 4);
                    e[0] = v;
                    e[32] = v;
                }
            }
        }
    }
    __syncthreads();

    // per-lane part of every table address (shared-window base included)
    const unsigned lane_base = unsigned(__cvta_generic_to_shared(table_raw)) +
                               unsigned(q * 256 + 4 * (rho + RPW * q));
    const unsigned sh = 4u * unsigned(rho);

    for (; rg < ngroups_rows; rg += nwarps) {
        const int64_t r = rg * RPW + rho;
        // next rows' loads before this row's lookups
        uint4 dn;
        float nn;
        cq2_load<CPR>(dn, nn, m, (rg + nwarps) * RPW + rho, q, g, nG);
        // rotate the 128-bit chunk right by 4*rho bits, then split every word
        // into its even nibbles (one per byte) and its odd nibbles
        unsigned w[4];
        w[0] = __funnelshift_r(d.x, d.y, sh);
        w[1] = __funnelshift_r(d.y, d.z, sh);
        w[2] = __funnelshift_r(d.z, d.w, sh);
        w[3] = __funnelshift_r(d.w, d.x, sh);
        float part0 = 0.0f, part1 = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const unsigned ev = w[i] & 0x0f0f0f0fu, od = (w[i] >> 4) & 0x0f0f0f0fu;
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int t = 8 * i + k;
                const unsigned nib = __byte_perm((k & 1) ? od : ev, 0u, 0x4440u | unsigned(k >> 1));
                const unsigned addr = nib * unsigned(NIB_STRIDE) + lane_base + 4u * unsigned(t);
                float tv;
                asm("ld.shared.f32 %0, [%1];" : "=f"(tv) : "r"(addr));
                if (k & 1)
                    part1 += tv;
                else
                    part0 += tv;
            }
        }
        const float part = part0 + part1;
        float acc = n * part;
#pragma unroll
        for (int dd = CPR / 2; dd >= 1; dd >>= 1) acc += __shfl_xor_sync(kFull, acc, dd);
        if (q == 0 && r < m.output) y[r] = acc;
        d = dn;
        n = nn;
    }
}

template <int CPR>
qmv_status launch_cq2_table(const qmv_cq_matrix &m, const float *p, float *y, cudaStream_t s) {
    const size_t smem = size_t(64) * CPR * 64;
    const void *kp = reinterpret_cast<const void *>(cq2_table_kernel<CPR>);
    if (!allow_smem(kp, smem)) return QMV_ERR_CUDA;
    const int64_t rgroups = (m.output + (32 / CPR) - 1) / (32 / CPR);
    int64_t blocks = (rgroups + 31) / 32;  // 32 warps per block
    if (blocks > sm_count()) blocks = sm_count();
    return from_cuda(launch_pdl(cq2_table_kernel<CPR>, dim3(unsigned(blocks)), dim3(1024), smem, s, m, p, y));
}

template <int B>
qmv_status launch_cq_general(const qmv_cq_matrix &m, const float *p, float *y, cudaStream_t s) {
    int blocks = grid_blocks(reinterpret_cast<const void *>(cq_matvec_general_kernel<B>), 256, 0, m.output);
    return from_cuda(launch_pdl(cq_matvec_general_kernel<B>, dim3(unsigned(blocks)), dim3(256), 0, s, m, p, y));
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

qmv_status launch_cq_matvec(const qmv_cq_matrix &m, const float *p, int batch, float *y,
                            cudaStream_t s) {
    const int64_t P = m.input_padded;
    const bool table_ok = m.bits == 2 && batch == 1 && m.group >= 64 &&
                          (P == 256 || P == 512 || P == 1024 || P == 2048) &&
                          (reinterpret_cast<uintptr_t>(m.packed) % 16) == 0;
    if (table_ok) {
        switch (P) {
            case 256: return launch_cq2_table<4>(m, p, y, s);
            case 512: return launch_cq2_table<8>(m, p, y, s);
            case 1024: return launch_cq2_table<16>(m, p, y, s);
            default: return launch_cq2_table<32>(m, p, y, s);
        }
    }
    switch (batch) {
        case 1: return launch_cq_general<1>(m, p, y, s);
        case 2: return launch_cq_general<2>(m, p, y, s);
        case 3: return launch_cq_general<3>(m, p, y, s);
        case 4: return launch_cq_general<4>(m, p, y, s);
        case 5: return launch_cq_general<5>(m, p, y, s);
        case 6: return launch_cq_general<6>(m, p, y, s);
        case 7: return launch_cq_general<7>(m, p, y, s);
        default: return launch_cq_general<8>(m, p, y, s);
    }
}

}  // namespace qmv
