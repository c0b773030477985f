// qmv_api.cu -- the extern "C" boundary of libqmv: argument validation,
// alias and overflow checks, then dispatch to the kernel launchers.
//
// Validation follows the loader discipline of the needle.js tutorial
// "Inference engine, part 1" (section 2 "Make bounds checks boring": check
// before every read, multiply shapes with overflow checks, never size work
// from unvalidated products; "Minimal tests": CQ packed length plus norm
// length must equal the record) and ds4f-disk issue #6, step 3 (refuse
// misaligned layouts).  No check reads device memory.
#include <stdint.h>
#include <string.h>

#include <climits>
#include <cmath>

#include <map>
#include <mutex>
#include <tuple>

#include "qmv_internal.h"

namespace qmv {

int sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

int occupancy(const void *kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    const auto key = std::make_tuple(kernel, dev, threads, smem);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
        per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = per_sm;
    return per_sm;
}

bool allow_smem(const void *kernel, size_t smem) {
    if (smem <= 48 * 1024) return true;
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(std::make_pair(kernel, dev));
    if (it != done.end() && it->second >= smem) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
        return false;
    done[std::make_pair(kernel, dev)] = smem;
    return true;
}

}  // namespace qmv

namespace {

// Sizes are capped well inside int64 so that every index product inside the
// kernels stays exact.
constexpr int64_t kMaxDim = int64_t(1) << 40;
constexpr int64_t kMaxBytes = int64_t(1) << 46;

bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a < 0 || b < 0) return false;
    if (__builtin_mul_overflow(a, b, out)) return false;
    return *out <= kMaxBytes;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Half-open byte ranges [a, a+na) and [b, b+nb) intersect.
bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    if (!a || !b || na <= 0 || nb <= 0) return false;
    uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + uint64_t(nb) && pb < pa + uint64_t(na);
}

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

// Shape checks shared by the three CQ entry points.
qmv_status check_cq_shape(const qmv_cq_matrix *m) {
    if (!m) return QMV_ERR_NULL;
    if (m->reserved != 0) return QMV_ERR_SHAPE;
    if (m->bits < 2 || m->bits > 5) return QMV_ERR_BITS;
    if (m->output < 0 || m->output > kMaxDim) return QMV_ERR_SHAPE;
    if (m->input_padded < 2 || m->input_padded > kMaxDim) return QMV_ERR_SHAPE;
    if (m->input < 1 || m->input > m->input_padded) return QMV_ERR_SHAPE;
    if (!is_pow2(m->group) || m->group < 2 || m->group > QMV_MAX_GROUP ||
        m->group > m->input_padded)
        return QMV_ERR_GROUP;
    if (m->input_padded % m->group != 0) return QMV_ERR_SHAPE;
    int64_t bits_total = 0;
    if (!mul_ok(m->input_padded, m->bits, &bits_total)) return QMV_ERR_OVERFLOW;
    if (m->row_bytes != (bits_total + 7) / 8) return QMV_ERR_SHAPE;
    int64_t tmp = 0;
    if (!mul_ok(m->output, m->row_bytes, &tmp)) return QMV_ERR_OVERFLOW;
    if (!mul_ok(m->output, (m->input_padded / m->group) * 2, &tmp)) return QMV_ERR_OVERFLOW;
    return QMV_OK;
}

qmv_status check_batch(int32_t batch) {
    return (batch < 1 || batch > QMV_MAX_BATCH) ? QMV_ERR_BATCH : QMV_OK;
}

// Byte sizes of the matrix arrays.
struct CqBytes {
    int64_t packed, norms, codebook;
};
CqBytes cq_bytes(const qmv_cq_matrix *m) {
    CqBytes b;
    b.packed = m->output * m->row_bytes;
    b.norms = m->output * (m->input_padded / m->group) * 2;
    b.codebook = (int64_t(1) << m->bits) * 4;
    return b;
}

qmv_status check_cq_data(const qmv_cq_matrix *m) {
    if (m->output > 0 && (!m->packed || !m->norms || !m->codebook)) return QMV_ERR_NULL;
    if (!aligned(m->norms, 2) || !aligned(m->codebook, 4)) return QMV_ERR_ALIGN;
    return QMV_OK;
}

// Checks shared by cq_matvec_multi and cq_prepare_matvec: the set's size, each
// matrix, the fields they must share, the output pointers, and that no output
// overlaps any matrix array, the activation `act` (act_bytes) or another output.
qmv_status check_cq_set(const qmv_cq_matrix *mats, int32_t nmats, int32_t batch, float *const *ys,
                        const void *act, int64_t act_bytes, const void *extra_out, int64_t extra_bytes) {
    if (!mats || !ys) return QMV_ERR_NULL;
    if (nmats < 1 || nmats > QMV_MAX_MATRICES) return QMV_ERR_SHAPE;
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    const qmv_cq_matrix &m0 = mats[0];
    int64_t yb[QMV_MAX_MATRICES];
    for (int i = 0; i < nmats; i++) {
        const qmv_cq_matrix &m = mats[i];
        if ((st = check_cq_shape(&m)) != QMV_OK) return st;
        if ((st = check_cq_data(&m)) != QMV_OK) return st;
        if (m.input != m0.input || m.input_padded != m0.input_padded || m.group != m0.group ||
            m.bits != m0.bits || m.row_bytes != m0.row_bytes || m.codebook != m0.codebook)
            return QMV_ERR_SHAPE;
        if (m.output > 0 && !ys[i]) return QMV_ERR_NULL;
        if (!aligned(ys[i], 4)) return QMV_ERR_ALIGN;
        if (!mul_ok(int64_t(batch) * 4, m.output, &yb[i])) return QMV_ERR_OVERFLOW;
    }
    for (int i = 0; i < nmats; i++) {
        if (overlaps(ys[i], yb[i], act, act_bytes) || overlaps(ys[i], yb[i], extra_out, extra_bytes))
            return QMV_ERR_ALIAS;
        for (int j = 0; j < nmats; j++) {
            const CqBytes b = cq_bytes(&mats[j]);
            if (overlaps(ys[i], yb[i], mats[j].packed, b.packed) ||
                overlaps(ys[i], yb[i], mats[j].norms, b.norms) ||
                overlaps(ys[i], yb[i], mats[j].codebook, b.codebook) ||
                overlaps(extra_out, extra_bytes, mats[j].packed, b.packed) ||
                overlaps(extra_out, extra_bytes, mats[j].norms, b.norms) ||
                overlaps(extra_out, extra_bytes, mats[j].codebook, b.codebook))
                return QMV_ERR_ALIAS;
            if (j != i && overlaps(ys[i], yb[i], ys[j], yb[j])) return QMV_ERR_ALIAS;
        }
    }
    if (overlaps(extra_out, extra_bytes, act, act_bytes)) return QMV_ERR_ALIAS;
    return QMV_OK;
}

int64_t cq_set_rows(const qmv_cq_matrix *mats, int32_t nmats) {
    int64_t rows = 0;
    for (int i = 0; i < nmats; i++) rows += mats[i].output;
    return rows;
}

// Checks of the sampler's own arguments.  ins[0..nin) are the call's inputs
// (u among them); y_out (y_out_bytes) is an output written before sampling,
// or NULL.  Outputs and workspace must be apart from every input and from
// each other.
qmv_status check_topk(int64_t R, int32_t batch, int32_t k, float temperature, const float *u,
                      const int64_t *top_index, const float *top_value, const float *top_prob,
                      const int64_t *token, const void *workspace, int64_t workspace_bytes,
                      const void *const *ins, const int64_t *inb, int nin, const void *y_out,
                      int64_t y_out_bytes) {
    if (R < 1) return QMV_ERR_SHAPE;
    if (R > INT32_MAX) return QMV_ERR_OVERFLOW;
    if (k < 1 || k > QMV_MAX_TOPK || k > R) return QMV_ERR_SHAPE;
    if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return QMV_ERR_ARG;
    if (!u || !top_index || !token || !workspace) return QMV_ERR_NULL;
    if (!aligned(u, 4) || !aligned(top_index, 8) || !aligned(top_value, 4) ||
        !aligned(top_prob, 4) || !aligned(token, 8) || !aligned(workspace, 16))
        return QMV_ERR_ALIGN;
    if (workspace_bytes < QMV_TOPK_WORKSPACE_BYTES) return QMV_ERR_SHAPE;
    const int64_t bk = int64_t(batch) * k;
    const void *outs[6] = {top_index, top_value, top_prob, token, workspace, y_out};
    const int64_t outb[6] = {bk * 8, top_value ? bk * 4 : 0, top_prob ? bk * 4 : 0,
                             int64_t(batch) * 8, workspace_bytes, y_out ? y_out_bytes : 0};
    for (int i = 0; i < 6; i++) {
        for (int j = 0; j < nin; j++)
            if (overlaps(outs[i], outb[i], ins[j], inb[j])) return QMV_ERR_ALIAS;
        for (int j = i + 1; j < 6; j++)
            if (overlaps(outs[i], outb[i], outs[j], outb[j])) return QMV_ERR_ALIAS;
    }
    return QMV_OK;
}

}  // namespace

extern "C" {

const char *qmv_status_string(qmv_status s) {
    switch (s) {
        case QMV_OK: return "QMV_OK";
        case QMV_ERR_NULL: return "QMV_ERR_NULL: a required pointer is NULL";
        case QMV_ERR_SHAPE: return "QMV_ERR_SHAPE: a size is out of range or inconsistent";
        case QMV_ERR_BITS: return "QMV_ERR_BITS: CQ bits must be 2, 3, 4 or 5";
        case QMV_ERR_GROUP:
            return "QMV_ERR_GROUP: CQ group must be a power of two in [2, min(input_padded, 32768)]";
        case QMV_ERR_BATCH: return "QMV_ERR_BATCH: batch must be in [1, 8]";
        case QMV_ERR_ALIGN: return "QMV_ERR_ALIGN: a pointer is not aligned to its element type";
        case QMV_ERR_OVERFLOW: return "QMV_ERR_OVERFLOW: a size product exceeds the library's limits";
        case QMV_ERR_ALIAS: return "QMV_ERR_ALIAS: an output overlaps an input";
        case QMV_ERR_CUDA: return "QMV_ERR_CUDA: the CUDA runtime reported an error";
        case QMV_ERR_ROW_ID: return "QMV_ERR_ROW_ID: a gathered row id was out of range";
        case QMV_ERR_ARG: return "QMV_ERR_ARG: a scalar argument is out of range";
    }
    return "unknown qmv_status";
}

int32_t qmv_abi_version(void) { return 1; }

qmv_status cq_prepare(const qmv_cq_matrix *m, const float *x, int32_t batch, float *prepared,
                      qmv_stream stream) {
    qmv_status st = check_cq_shape(m);
    if (st != QMV_OK) return st;
    if ((st = check_batch(batch)) != QMV_OK) return st;
    if (!x || !prepared) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(prepared, 4)) return QMV_ERR_ALIGN;
    int64_t xb = 0, pb = 0;
    if (!mul_ok(int64_t(batch) * 4, m->input, &xb) || !mul_ok(int64_t(batch) * 4, m->input_padded, &pb))
        return QMV_ERR_OVERFLOW;
    if (overlaps(prepared, pb, x, xb)) return QMV_ERR_ALIAS;
    return qmv::launch_cq_prepare(*m, x, batch, prepared, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status cq_matvec(const qmv_cq_matrix *m, const float *prepared, int32_t batch, float *y,
                     qmv_stream stream) {
    qmv_status st = check_cq_shape(m);
    if (st != QMV_OK) return st;
    if ((st = check_batch(batch)) != QMV_OK) return st;
    if ((st = check_cq_data(m)) != QMV_OK) return st;
    if (!prepared || (m->output > 0 && !y)) return QMV_ERR_NULL;
    if (!aligned(prepared, 4) || !aligned(y, 4)) return QMV_ERR_ALIGN;
    int64_t pb = 0, yb = 0;
    if (!mul_ok(int64_t(batch) * 4, m->input_padded, &pb) || !mul_ok(int64_t(batch) * 4, m->output, &yb))
        return QMV_ERR_OVERFLOW;
    CqBytes b = cq_bytes(m);
    if (overlaps(y, yb, prepared, pb) || overlaps(y, yb, m->packed, b.packed) ||
        overlaps(y, yb, m->norms, b.norms) || overlaps(y, yb, m->codebook, b.codebook))
        return QMV_ERR_ALIAS;
    if (m->output == 0) return QMV_OK;
    return qmv::launch_cq_matvec(*m, prepared, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status cq_matvec_multi(const qmv_cq_matrix *mats, int32_t nmats, const float *prepared,
                           int32_t batch, float *const *ys, qmv_stream stream) {
    if (!prepared) return QMV_ERR_NULL;
    if (!aligned(prepared, 4)) return QMV_ERR_ALIGN;
    if (!mats) return QMV_ERR_NULL;
    int64_t pb = 0;
    if (nmats >= 1 && !mul_ok(int64_t(batch < 1 ? 1 : batch) * 4, mats[0].input_padded, &pb))
        return QMV_ERR_OVERFLOW;
    qmv_status st = check_cq_set(mats, nmats, batch, ys, prepared, pb, nullptr, 0);
    if (st != QMV_OK) return st;
    if (cq_set_rows(mats, nmats) == 0) return QMV_OK;
    return qmv::launch_cq_set(mats, nmats, prepared, nullptr, nullptr, batch, ys,
                              reinterpret_cast<cudaStream_t>(stream));
}

qmv_status cq_prepare_matvec(const qmv_cq_matrix *mats, int32_t nmats, const float *x, int32_t batch,
                             float *prepared, float *const *ys, qmv_stream stream) {
    if (!x) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(prepared, 4)) return QMV_ERR_ALIGN;
    if (!mats) return QMV_ERR_NULL;
    int64_t xb = 0, pb = 0;
    if (nmats >= 1 && (!mul_ok(int64_t(batch < 1 ? 1 : batch) * 4, mats[0].input, &xb) ||
                       !mul_ok(int64_t(batch < 1 ? 1 : batch) * 4, mats[0].input_padded, &pb)))
        return QMV_ERR_OVERFLOW;
    qmv_status st = check_cq_set(mats, nmats, batch, ys, x, xb, prepared, prepared ? pb : 0);
    if (st != QMV_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (qmv::cq_fused_fits(mats[0], batch)) {
        if (cq_set_rows(mats, nmats) == 0) {
            // no matrix rows: the prepared activation is still produced on request
            return prepared ? qmv::launch_cq_prepare(mats[0], x, batch, prepared, s) : QMV_OK;
        }
        return qmv::launch_cq_set(mats, nmats, nullptr, x, prepared, batch, ys, s);
    }
    // too wide to prepare on chip: two launches through the prepared vector
    if (!prepared) return QMV_ERR_NULL;
    st = qmv::launch_cq_prepare(mats[0], x, batch, prepared, s);
    if (st != QMV_OK || cq_set_rows(mats, nmats) == 0) return st;
    return qmv::launch_cq_set(mats, nmats, prepared, nullptr, nullptr, batch, ys, s);
}

qmv_status cq_dequantize_row(const qmv_cq_matrix *m, const int32_t *rows, int64_t n, float *out,
                             int32_t *dev_status, qmv_stream stream) {
    qmv_status st = check_cq_shape(m);
    if (st != QMV_OK) return st;
    if (n < 0 || n > kMaxDim) return QMV_ERR_SHAPE;
    if (n == 0) return QMV_OK;
    if ((st = check_cq_data(m)) != QMV_OK) return st;
    if (!rows || !out) return QMV_ERR_NULL;
    if (!aligned(rows, 4) || !aligned(out, 4) || !aligned(dev_status, 4)) return QMV_ERR_ALIGN;
    int64_t ob = 0;
    if (!mul_ok(n * 4, m->input, &ob)) return QMV_ERR_OVERFLOW;
    CqBytes b = cq_bytes(m);
    if (overlaps(out, ob, rows, n * 4) || overlaps(out, ob, m->packed, b.packed) ||
        overlaps(out, ob, m->norms, b.norms) || overlaps(out, ob, m->codebook, b.codebook) ||
        overlaps(out, ob, dev_status, 4))
        return QMV_ERR_ALIAS;
    if (dev_status && (overlaps(dev_status, 4, rows, n * 4) ||
                       overlaps(dev_status, 4, m->packed, b.packed) ||
                       overlaps(dev_status, 4, m->norms, b.norms) ||
                       overlaps(dev_status, 4, m->codebook, b.codebook)))
        return QMV_ERR_ALIAS;
    return qmv::launch_cq_dequantize_row(*m, rows, n, out, dev_status,
                                         reinterpret_cast<cudaStream_t>(stream));
}

qmv_status f8_matvec_argmax(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                            int64_t SC, const float *x, int32_t batch, float *y, int64_t *out_index,
                            float *out_value, void *workspace, int64_t workspace_bytes,
                            qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 1 || R > kMaxDim || C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    if (SR < 1 || SR > R || SC < 1 || SC > C) return QMV_ERR_SHAPE;
    int64_t wb = 0, sb = 0, xb = 0, yb = 0, t = 0;
    if (!mul_ok(R, C, &wb) || !mul_ok(SR, SC, &sb) || !mul_ok(int64_t(batch) * 4, C, &xb) ||
        !mul_ok(int64_t(batch) * 4, R, &yb) || !mul_ok(R, SR, &t) || !mul_ok(C, SC, &t))
        return QMV_ERR_OVERFLOW;
    if (!w || !scale || !x || !out_index || !out_value || !workspace) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(y, 4) || !aligned(out_index, 8) || !aligned(out_value, 4) ||
        !aligned(workspace, 16))
        return QMV_ERR_ALIGN;
    if (workspace_bytes < QMV_F8_ARGMAX_WORKSPACE_BYTES(batch)) return QMV_ERR_SHAPE;
    const int64_t ib = int64_t(batch) * 8, vb = int64_t(batch) * 4, kb = workspace_bytes;
    // every output (and the workspace) apart from every input and each other
    const void *outs[4] = {y, out_index, out_value, workspace};
    const int64_t outb[4] = {y ? yb : 0, ib, vb, kb};
    const void *ins[3] = {w, scale, x};
    const int64_t inb[3] = {wb, sb, xb};
    for (int i = 0; i < 4; i++) {
        for (int j = 0; j < 3; j++)
            if (overlaps(outs[i], outb[i], ins[j], inb[j])) return QMV_ERR_ALIAS;
        for (int j = i + 1; j < 4; j++)
            if (overlaps(outs[i], outb[i], outs[j], outb[j])) return QMV_ERR_ALIAS;
    }
    return qmv::launch_f8_matvec_argmax(w, R, C, scale, SR, SC, x, batch, y, out_index, out_value,
                                        workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status i8_matvec(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale, const float *x,
                     int32_t batch, float *y, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 0 || R > kMaxDim || C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    int64_t wb = 0, sb = 0, xb = 0, yb = 0;
    if (!mul_ok(R, C, &wb) || !mul_ok(R, (C + 15) / 16, &sb) || !mul_ok(int64_t(batch) * 4, C, &xb) ||
        !mul_ok(int64_t(batch) * 4, R, &yb))
        return QMV_ERR_OVERFLOW;
    if (!x) return QMV_ERR_NULL;
    if (R > 0 && (!w || !scale || !y)) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(y, 4)) return QMV_ERR_ALIGN;
    if (overlaps(y, yb, w, wb) || overlaps(y, yb, scale, sb) || overlaps(y, yb, x, xb))
        return QMV_ERR_ALIAS;
    if (R == 0) return QMV_OK;
    return qmv::launch_i8_matvec(w, R, C, scale, x, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status i8_quantize_x(const float *x, int64_t C, int32_t batch, int8_t *xq, float *xscale,
                         qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    int64_t xb = 0, qb = 0, db = 0;
    if (!mul_ok(int64_t(batch) * 4, C, &xb) || !mul_ok(int64_t(batch), C, &qb) ||
        !mul_ok(int64_t(batch) * 4, (C + 31) / 32, &db))
        return QMV_ERR_OVERFLOW;
    if (!x || !xq || !xscale) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(xscale, 4)) return QMV_ERR_ALIGN;
    if (overlaps(xq, qb, x, xb) || overlaps(xscale, db, x, xb) || overlaps(xq, qb, xscale, db))
        return QMV_ERR_ALIAS;
    return qmv::launch_i8_quantize_x(x, C, batch, xq, xscale, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status i8_matvec_q8(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale, const int8_t *xq,
                        const float *xscale, int32_t batch, float *y, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 0 || R > kMaxDim || C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    int64_t wb = 0, sb = 0, qb = 0, db = 0, yb = 0;
    if (!mul_ok(R, C, &wb) || !mul_ok(R, (C + 15) / 16, &sb) || !mul_ok(int64_t(batch), C, &qb) ||
        !mul_ok(int64_t(batch) * 4, (C + 31) / 32, &db) || !mul_ok(int64_t(batch) * 4, R, &yb))
        return QMV_ERR_OVERFLOW;
    if (!xq || !xscale) return QMV_ERR_NULL;
    if (R > 0 && (!w || !scale || !y)) return QMV_ERR_NULL;
    if (!aligned(xscale, 4) || !aligned(y, 4)) return QMV_ERR_ALIGN;
    if (overlaps(y, yb, w, wb) || overlaps(y, yb, scale, sb) || overlaps(y, yb, xq, qb) ||
        overlaps(y, yb, xscale, db))
        return QMV_ERR_ALIAS;
    if (R == 0) return QMV_OK;
    return qmv::launch_i8_matvec_q8(w, R, C, scale, xq, xscale, batch, y,
                                    reinterpret_cast<cudaStream_t>(stream));
}

qmv_status hadamard_mlp(const float *x, int64_t n, int64_t D, const float *d1, const float *d2,
                        const float *d3, const float *residual, const float *u, int32_t batch,
                        float *out, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (D < 1 || D > QMV_MAX_HADAMARD || (D & (D - 1)) != 0 || n < 1 || n > D) return QMV_ERR_SHAPE;
    if (!x || !d1 || !d2 || !d3 || !out) return QMV_ERR_NULL;
    const float *in[] = {x, d1, d2, d3, residual, u};
    for (const float *p : in)
        if (p && !aligned(p, 4)) return QMV_ERR_ALIGN;
    if (!aligned(out, 4)) return QMV_ERR_ALIGN;
    const int64_t vb = int64_t(batch) * n * 4, db = D * 4;
    if (overlaps(out, vb, x, vb) || overlaps(out, vb, d1, db) || overlaps(out, vb, d2, db) ||
        overlaps(out, vb, d3, db) || (residual && overlaps(out, vb, residual, vb)) ||
        (u && overlaps(out, vb, u, vb)))
        return QMV_ERR_ALIAS;
    return qmv::launch_hadamard_mlp(x, n, int(D), d1, d2, d3, residual, u, batch, out,
                                    1.0 / std::sqrt(double(D)), reinterpret_cast<cudaStream_t>(stream));
}

qmv_status f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale, int64_t SR,
                     int64_t SC, const float *x, int32_t batch, float *y, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 0 || R > kMaxDim || C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    if (SR < 1 || SR > (R > 0 ? R : 1) || SC < 1 || SC > C) return QMV_ERR_SHAPE;
    int64_t wb = 0, sb = 0, xb = 0, yb = 0, t = 0;
    if (!mul_ok(R, C, &wb) || !mul_ok(SR, SC, &sb) || !mul_ok(int64_t(batch) * 4, C, &xb) ||
        !mul_ok(int64_t(batch) * 4, R, &yb))
        return QMV_ERR_OVERFLOW;
    // the kernels form r * SR and c * SC in 64 bits
    if (!mul_ok(R, SR, &t) || !mul_ok(C, SC, &t)) return QMV_ERR_OVERFLOW;
    if (!x || !scale) return QMV_ERR_NULL;
    if (R > 0 && (!w || !y)) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(y, 4)) return QMV_ERR_ALIGN;
    if (overlaps(y, yb, w, wb) || overlaps(y, yb, scale, sb) || overlaps(y, yb, x, xb))
        return QMV_ERR_ALIAS;
    if (R == 0) return QMV_OK;
    return qmv::launch_f8_matvec(w, R, C, scale, SR, SC, x, batch, y,
                                 reinterpret_cast<cudaStream_t>(stream));
}

qmv_status topk_sample(const float *y, int64_t R, int32_t batch, int32_t k, float temperature,
                       const float *u, int64_t *top_index, float *top_value, float *top_prob,
                       int64_t *token, void *workspace, int64_t workspace_bytes, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 1) return QMV_ERR_SHAPE;
    if (R > INT32_MAX) return QMV_ERR_OVERFLOW;
    if (!y) return QMV_ERR_NULL;
    if (!aligned(y, 4)) return QMV_ERR_ALIGN;
    const void *ins[2] = {y, u};
    const int64_t inb[2] = {int64_t(batch) * R * 4, int64_t(batch) * 4};
    st = check_topk(R, batch, k, temperature, u, top_index, top_value, top_prob, token, workspace,
                    workspace_bytes, ins, inb, 2, nullptr, 0);
    if (st != QMV_OK) return st;
    return qmv::launch_topk_sample(y, R, batch, k, temperature, u, top_index, top_value, top_prob,
                                   token, workspace, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status f8_matvec_topk_sample(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                                 int64_t SR, int64_t SC, const float *x, int32_t batch, float *y,
                                 int32_t k, float temperature, const float *u, int64_t *top_index,
                                 float *top_value, float *top_prob, int64_t *token,
                                 void *workspace, int64_t workspace_bytes, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 1 || R > kMaxDim || C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    if (SR < 1 || SR > R || SC < 1 || SC > C) return QMV_ERR_SHAPE;
    int64_t wb = 0, sb = 0, xb = 0, yb = 0, t = 0;
    if (!mul_ok(R, C, &wb) || !mul_ok(SR, SC, &sb) || !mul_ok(int64_t(batch) * 4, C, &xb) ||
        !mul_ok(int64_t(batch) * 4, R, &yb) || !mul_ok(R, SR, &t) || !mul_ok(C, SC, &t))
        return QMV_ERR_OVERFLOW;
    if (!w || !scale || !x || !y) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(y, 4)) return QMV_ERR_ALIGN;
    const void *ins[4] = {w, scale, x, u};
    const int64_t inb[4] = {wb, sb, xb, int64_t(batch) * 4};
    st = check_topk(R, batch, k, temperature, u, top_index, top_value, top_prob, token, workspace,
                    workspace_bytes, ins, inb, 4, y, yb);
    if (st != QMV_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = qmv::launch_f8_matvec(w, R, C, scale, SR, SC, x, batch, y, s);
    if (st != QMV_OK) return st;
    return qmv::launch_topk_sample(y, R, batch, k, temperature, u, top_index, top_value, top_prob,
                                   token, workspace, s);
}

qmv_status i8_matvec_topk_sample(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                                 const float *x, int32_t batch, float *y, int32_t k,
                                 float temperature, const float *u, int64_t *top_index,
                                 float *top_value, float *top_prob, int64_t *token,
                                 void *workspace, int64_t workspace_bytes, qmv_stream stream) {
    qmv_status st = check_batch(batch);
    if (st != QMV_OK) return st;
    if (R < 1 || R > kMaxDim || C < 1 || C > kMaxDim) return QMV_ERR_SHAPE;
    int64_t wb = 0, sb = 0, xb = 0, yb = 0;
    if (!mul_ok(R, C, &wb) || !mul_ok(R, (C + 15) / 16, &sb) || !mul_ok(int64_t(batch) * 4, C, &xb) ||
        !mul_ok(int64_t(batch) * 4, R, &yb))
        return QMV_ERR_OVERFLOW;
    if (!w || !scale || !x || !y) return QMV_ERR_NULL;
    if (!aligned(x, 4) || !aligned(y, 4)) return QMV_ERR_ALIGN;
    const void *ins[4] = {w, scale, x, u};
    const int64_t inb[4] = {wb, sb, xb, int64_t(batch) * 4};
    st = check_topk(R, batch, k, temperature, u, top_index, top_value, top_prob, token, workspace,
                    workspace_bytes, ins, inb, 4, y, yb);
    if (st != QMV_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = qmv::launch_i8_matvec(w, R, C, scale, x, batch, y, s);
    if (st != QMV_OK) return st;
    return qmv::launch_topk_sample(y, R, batch, k, temperature, u, top_index, top_value, top_prob,
                                   token, workspace, s);
}

qmv_status qmv_tc_wait_timeouts(uint64_t *count) {
    if (!count) return QMV_ERR_NULL;
    unsigned long long c = 0;
    const qmv_status st = qmv::f8_tc_wait_timeouts(&c);
    if (st == QMV_OK) *count = uint64_t(c);
    return st;
}

}  // extern "C"
