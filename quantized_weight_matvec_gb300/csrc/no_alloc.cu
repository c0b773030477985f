// no_alloc.cu -- f8_matvec_argmax_noalloc: the fused head matvec + greedy
// selection for callers that cannot allocate device memory.
//
// f8_matvec_argmax needs a small scratch buffer (an arrival counter and one
// partial result per block and vector) that its caller provides.  Some callers have no way to
// get one: an engine that has handed the whole device to its own memory pool
// at start-up and treats any further cudaMalloc as an error, or a plug-in
// interface that passes tensors in and out but offers no workspace and no
// allocator.  For them this entry point takes its scratch from a fixed array
// that lives in the library itself, so it never allocates.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds its 256 KiB (and 16 bytes) until the process exits.  In host code its
// name is only a host-side stand-in for the device symbol, not a device
// address, so the device address is looked up once per device with
// cudaGetSymbolAddress (while that device is current) and passed to the
// kernels like any other workspace pointer.
#include <cuda.h>

#include <mutex>

#include "qmv_internal.h"

namespace {

// Enough for every launch the argmax kernels make: the arrival counter and
// at most QMV_ARGMAX_MAX_BLOCKS blocks x QMV_MAX_BATCH vectors x 16 bytes.
// A __device__ array starts zeroed, so the counter is ready for the first
// call, and every call leaves it zero.
constexpr size_t kScratchBytes = size_t(QMV_F8_ARGMAX_WORKSPACE_BYTES(QMV_MAX_BATCH));

static __device__ __align__(256) unsigned char g_argmax_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current CUDA context (the device's
// primary context under the runtime), or 0 when the driver cannot say.  A
// context that is destroyed and created again (cudaDeviceReset, a primary
// context reset) gets a new id, so an address cached under the old id is
// never reused.  The driver functions are fetched through the runtime, so the
// library needs no link against the driver library.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(fn);
        (void)cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_argmax_scratch in the current context.  It is looked
// up with cudaGetSymbolAddress on the first call made in each context (with
// the device current; the lookup initialises the device's primary context if
// nothing has yet) and cached under the context's id; while the id cannot be
// read (no context yet, or an old driver) it is looked up on every call.
void *scratch_address(qmv_status *status) {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = QMV_ERR_CUDA;
        return nullptr;
    }
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || id == 0 || ctx_of[dev] != id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_argmax_scratch) != cudaSuccess || !p) {
            *status = QMV_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
        ctx_of[dev] = id;
    }
    *status = QMV_OK;
    return addr[dev];
}

}  // namespace

extern "C" qmv_status f8_matvec_argmax_noalloc(const uint8_t *w, int64_t R, int64_t C,
                                               const uint8_t *scale, int64_t SR, int64_t SC,
                                               const float *x, int32_t batch, float *y,
                                               int64_t *out_index, float *out_value,
                                               qmv_stream stream) {
    // The scratch holds QMV_MAX_BATCH vectors' partials; larger batches are
    // refused (the regular entry point refuses them too).
    if (batch < 1 || batch > QMV_MAX_BATCH ||
        QMV_F8_ARGMAX_WORKSPACE_BYTES(batch) > int64_t(kScratchBytes))
        return QMV_ERR_BATCH;
    qmv_status st = QMV_OK;
    void *ws = scratch_address(&st);
    if (st != QMV_OK) return st;
    // All checks of the regular entry point still apply.
    return f8_matvec_argmax(w, R, C, scale, SR, SC, x, batch, y, out_index, out_value, ws,
                            int64_t(kScratchBytes), stream);
}
