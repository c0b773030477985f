// mlp_kernels.cu -- the Hadamard MLP block, sm_103a.
//
// Method: needle.js tutorial "Inference engine, part 2: kernels and token
// step", section 8 ("Hadamard MLP"), from the padded normalised block input:
//
//   z = pad(x, D); z *= d1; normalizedFwht(z); z[i] = silu(d2[i] * z[i]);
//   normalizedFwht(z); z *= d3; out = (residual + z[0..n)) - u
//
// normalizedFwht is the section-1 butterfly over the whole length D followed
// by the product with 1/sqrt(D) in float64, rounded to float32 (as prepare,
// section 2).  Every stored value is a float32, as in the page's
// Float32Array: the diagonal products, each butterfly result, the scaled
// values, the residual sum and the update difference are single rounded
// float32 operations, so they are bit-identical to that staging.  silu is
// evaluated in float32 (v / (1 + e^-v) with expf and an IEEE divide) from
// the float32 product d2 * z; the page evaluates it in float64, so results
// agree within a few float32 ulps of each silu value, not bit for bit.
//
// One block per vector.  Thread t holds E consecutive elements (t*E ..
// t*E+E-1).  Strides below 32E run in registers and warp shuffles
// (fwht_warp); the remaining strides run on a shared-memory copy of the
// vector, one barrier per stride.
#include <stdint.h>

#include "fwht_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

struct MlpArgs {
    const float *x, *d1, *d2, *d3, *res, *u;
    float *out;
    int64_t n;
    int D;
    Scale s;  // RN64(1/sqrt(D)), and its float32 split
};

// Whole-vector FWHT: v holds elements tid*E .. tid*E+E-1 of the D values.
template <int E>
__device__ __forceinline__ void fwht_block(float (&v)[E], float *sm, int D, int tid, int nt) {
    const int span = 32 * E;
    if (D <= span) {
        fwht_warp<E>(v, D, tid & 31);
        return;
    }
    fwht_warp<E>(v, span, tid & 31);
    __syncthreads();  // a previous pass may still be reading sm
#pragma unroll
    for (int e = 0; e < E; e++) sm[tid * E + e] = v[e];
    for (int h = span; h < D; h <<= 1) {
        __syncthreads();
        for (int t = tid; t < D / 2; t += nt) {
            const int i = ((t & ~(h - 1)) << 1) | (t & (h - 1));
            const float a = sm[i], b = sm[i + h];
            sm[i] = __fadd_rn(a, b);
            sm[i + h] = __fsub_rn(a, b);
        }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; e++) v[e] = sm[tid * E + e];
}

__device__ __forceinline__ float silu32(float a) {
    return __fdiv_rn(a, __fadd_rn(1.0f, expf(-a)));
}

// PRE: the diagonals d2, d3 and the residual / u values are loaded with x
// and d1 at the start, so their latency overlaps the first transform.
template <int E, bool PRE>
__global__ void __launch_bounds__(1024) hadamard_mlp_kernel(MlpArgs a) {
    extern __shared__ float sm[];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t j = blockIdx.x;
    const int i0 = tid * E;
    const bool live = i0 < a.D;  // only false when D < 32 (one partial warp)
    const float *xv = a.x + j * a.n;
    const float *rv = a.res ? a.res + j * a.n : nullptr;
    const float *uv = a.u ? a.u + j * a.n : nullptr;
    float v[E], g2[E], g3[E], rr[E], uu[E];
#pragma unroll
    for (int e = 0; e < E; e++) {
        const int i = i0 + e;
        const float xe = (live && i < a.n) ? __ldg(xv + i) : 0.0f;
        v[e] = live ? __fmul_rn(xe, __ldg(a.d1 + i)) : 0.0f;
        if (PRE) {
            g2[e] = live ? __ldg(a.d2 + i) : 0.0f;
            g3[e] = live ? __ldg(a.d3 + i) : 0.0f;
            rr[e] = (rv && live && i < a.n) ? __ldg(rv + i) : 0.0f;
            uu[e] = (uv && live && i < a.n) ? __ldg(uv + i) : 0.0f;
        }
    }
    fwht_block<E>(v, sm, a.D, tid, nt);
    scale_rn_all<E>(v, a.s);
#pragma unroll
    for (int e = 0; e < E; e++) {
        const float d2e = PRE ? g2[e] : (live ? __ldg(a.d2 + i0 + e) : 0.0f);
        v[e] = silu32(__fmul_rn(d2e, v[e]));
    }
    fwht_block<E>(v, sm, a.D, tid, nt);
    scale_rn_all<E>(v, a.s);
    float *ov = a.out + j * a.n;
#pragma unroll
    for (int e = 0; e < E; e++) {
        const int i = i0 + e;
        if (!live || i >= a.n) continue;
        const float d3e = PRE ? g3[e] : __ldg(a.d3 + i);
        float o = __fmul_rn(v[e], d3e);
        if (rv) o = __fadd_rn(PRE ? rr[e] : __ldg(rv + i), o);
        if (uv) o = __fsub_rn(o, PRE ? uu[e] : __ldg(uv + i));
        ov[i] = o;
    }
}

template <int E>
qmv_status launch_mlp(const MlpArgs &a, int batch, cudaStream_t s) {
    constexpr bool PRE = (E <= 8);
    const int nt = a.D >= 32 * E ? a.D / E : 32;
    const size_t smem = a.D > 32 * E ? size_t(a.D) * sizeof(float) : 0;
    auto kern = hadamard_mlp_kernel<E, PRE>;
    if (smem > 48 * 1024 && !allow_smem(reinterpret_cast<const void *>(kern), smem)) return QMV_ERR_CUDA;
    return from_cuda(launch_pdl(kern, dim3(unsigned(batch)), dim3(unsigned(nt)), smem, s, a));
}

}  // namespace

qmv_status launch_hadamard_mlp(const float *x, int64_t n, int D, const float *d1, const float *d2,
                               const float *d3, const float *residual, const float *u, int batch,
                               float *out, double s, cudaStream_t stream) {
    const MlpArgs a{x, d1, d2, d3, residual, u, out, n, D, make_scale(s)};
    // E values per thread: one warp up to D = 256, then 8 per thread up to
    // 1024 threads (D = 8192), then 16 and 32.
    if (D <= 32) return launch_mlp<1>(a, batch, stream);
    if (D == 64) return launch_mlp<2>(a, batch, stream);
    if (D == 128) return launch_mlp<4>(a, batch, stream);
    if (D <= 8192) return launch_mlp<8>(a, batch, stream);
    if (D == 16384) return launch_mlp<16>(a, batch, stream);
    return launch_mlp<32>(a, batch, stream);
}

}  // namespace qmv
