// qmv_internal.h -- host-side interfaces between the C-ABI layer (qmv_api.cu)
// and the kernel translation units (cq_kernels.cu, f8_kernels.cu).
// Arguments reaching these launchers are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/qmv.h"

namespace qmv {

// Number of SMs of the current device (cached per device).
int sm_count();

// Resident blocks per SM of `kernel` at (threads, dynamic smem) on the
// current device; cached per (kernel, device, threads, smem).  Returns >= 1.
int occupancy(const void *kernel, int threads, size_t smem);

// Raises the kernel's dynamic shared-memory limit to `smem` bytes once per
// (kernel, device).  Returns false if the runtime refuses.
bool allow_smem(const void *kernel, size_t smem);

// Blocks for a grid of `threads`-thread blocks that covers `warps_wanted`
// warps, capped at resident_per_sm * SMs.
inline int grid_blocks(const void *kernel, int threads, size_t smem, int64_t warps_wanted) {
    const int64_t cap = int64_t(occupancy(kernel, threads, smem)) * sm_count();
    int64_t need = (warps_wanted * 32 + threads - 1) / threads;
    if (need < 1) need = 1;
    return int(need < cap ? need : cap);
}

// Programmatic dependent launch.  pdl_wait() returns once all work that
// precedes the kernel in the stream has completed and its memory is
// visible.  Launched with launch_pdl(), a kernel may be scheduled while the
// previous kernel in the stream is still running (once that kernel has
// called pdl_trigger()), which hides the launch latency between the
// back-to-back calls of a decode step.  Every kernel of the library reads
// activations and writes outputs only after pdl_wait(), so stream order holds
// for them whatever the preceding kernel is.  The matrices are model
// weights, read-only for the library's calls: most matvec kernels (CQ, F8,
// I8) load their first weights before pdl_wait(), so a matrix must not be
// written by kernels still queued ahead of a call on its stream (see qmv.h).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Fills a cudaError_t into a qmv_status.
inline qmv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMV_OK : QMV_ERR_CUDA; }

// ---- CQ ------------------------------------------------------------------
qmv_status launch_cq_prepare(const qmv_cq_matrix &m, const float *x, int batch, float *prepared,
                             cudaStream_t s);
qmv_status launch_cq_dequantize_row(const qmv_cq_matrix &m, const int32_t *rows, int64_t n,
                                    float *out, int32_t *dev_status, cudaStream_t s);
qmv_status launch_cq_matvec(const qmv_cq_matrix &m, const float *prepared, int batch, float *y,
                            cudaStream_t s);
// Several matrices sharing input width, group, bits and codebook.  With x
// non-NULL the activation is prepared inside the launch (and also stored to
// prepared_out when that is non-NULL); otherwise p is the prepared vector.
qmv_status launch_cq_set(const qmv_cq_matrix *mats, int nmats, const float *p, const float *x,
                         float *prepared_out, int batch, float *const *ys, cudaStream_t s);
// Whether cq_prepare_matvec can prepare on chip (else it runs two launches).
bool cq_fused_fits(const qmv_cq_matrix &m, int batch);

// ---- I8 ------------------------------------------------------------------
qmv_status launch_i8_matvec(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                            const float *x, int batch, float *y, cudaStream_t s);

// ---- I8 over int8 activations (i8q_kernels.cu) --------------------------------
qmv_status launch_i8_quantize_x(const float *x, int64_t C, int batch, int8_t *xq, float *xd,
                                cudaStream_t s);
qmv_status launch_i8_matvec_q8(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                               const int8_t *xq, const float *xd, int batch, float *y,
                               cudaStream_t s);
// The I8 tensor-core kernel over q * d activations (i8_kernels.cu): false when
// it does not take the call (batch < 2, C not a multiple of 64 in
// [256, 4096], unaligned w or xq); else launches it and sets st.
bool launch_i8_matvec_q8_mma(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                             const int8_t *xq, const float *xd, int batch, float *y, cudaStream_t s,
                             qmv_status &st);

// ---- Hadamard MLP ----------------------------------------------------------
qmv_status launch_hadamard_mlp(const float *x, int64_t n, int D, const float *d1, const float *d2,
                               const float *d3, const float *residual, const float *u, int batch,
                               float *out, double s, cudaStream_t stream);

// ---- F8 ------------------------------------------------------------------
qmv_status launch_f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                            int64_t SR, int64_t SC, const float *x, int batch, float *y,
                            cudaStream_t s);
qmv_status launch_f8_matvec_argmax(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                                   int64_t SR, int64_t SC, const float *x, int batch, float *y,
                                   int64_t *out_index, float *out_value, void *workspace,
                                   int64_t workspace_bytes, cudaStream_t s);
// Waits of the fifth-generation tensor-core F8 kernel that ran out of time
// (f8_tc_kernels.cu).
qmv_status f8_tc_wait_timeouts(unsigned long long *count);


// ---- top-k sampling ----------------------------------------------------------
// Slices per vector of the first selection pass (1 means a single launch).
int topk_slices(int64_t R, int batch);
qmv_status launch_topk_sample(const float *y, int64_t R, int batch, int k, float temperature,
                              const float *u, int64_t *top_index, float *top_value, float *top_prob,
                              int64_t *token, void *workspace, cudaStream_t s);

}  // namespace qmv
