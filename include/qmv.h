/*
 * qmv.h -- C ABI of libqmv, the GB300 (sm_103a) quantized-weight matvec.
 *
 * Two weight formats, each applied to 1..8 activation vectors at once:
 *
 *   CQ  (needle.js tutorial "Inference engine, part 2: kernels and token
 *        step", sections 1-3 and "Row gather"; matrix layout from "part 1:
 *        loader and tokenizer", section 4 "Retain packed matrices"):
 *        activations are zero-padded and rotated by a per-group Walsh-
 *        Hadamard transform; weights are 2/3/4/5-bit codebook indices with
 *        one binary16 norm per (row, group).
 *   F8  (ds4f-disk issue #6 "attention + tokenizer + sampling", work item 1
 *        and step 1): E4M3 weight bytes with E8M0 block scales.
 *
 * Conventions shared by every entry point
 *   - All array pointers are DEVICE pointers, owned by the caller.  The
 *     library allocates nothing, never synchronises the device and never
 *     reads device memory on the host.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream of the current device).
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns its status and launches nothing.  Outputs are
 *     then left untouched.
 *   - Arrays are dense and row-major, batch-major for activations:
 *     x[v][k] lives at x + v * width + k.
 *   - Outputs are fully overwritten and must not overlap any input
 *     (QMV_ERR_ALIAS).  Repeated calls on equal inputs give bitwise equal
 *     outputs (fixed reduction order, no floating-point atomics).
 *   - float pointers must be 4-byte aligned, binary16 pointers 2-byte
 *     aligned, int32 pointers 4-byte aligned (QMV_ERR_ALIGN).  Wider
 *     alignment and shapes that are multiples of 16 bytes let the library
 *     pick its vectorised kernels; other layouts take a general kernel
 *     with the same results.
 *   - Errors of the CUDA runtime at launch are reported as QMV_ERR_CUDA.
 *   - Calls may start on the GPU before the kernel queued just ahead of them
 *     on the same stream has finished (programmatic dependent launch).
 *     Activations are read and outputs written only once everything ahead
 *     in the stream has completed.  Weight matrices are treated as
 *     read-only model weights and may be read earlier: write a matrix with
 *     a copy, or with a kernel followed by a stream or event
 *     synchronisation, before its first use -- never with a kernel still
 *     queued ahead of the call on the same stream.
 */
#ifndef QMV_H
#define QMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QMV_API __attribute__((visibility("default")))
#else
#define QMV_API
#endif

/* Same handle type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *qmv_stream;

typedef enum {
    QMV_OK = 0,
    QMV_ERR_NULL = 1,      /* a required pointer is NULL                         */
    QMV_ERR_SHAPE = 2,     /* a size is out of range or inconsistent             */
    QMV_ERR_BITS = 3,      /* CQ bits not in {2, 3, 4, 5}                        */
    QMV_ERR_GROUP = 4,     /* CQ group not a power of two in [2, min(P, 32768)]   */
    QMV_ERR_BATCH = 5,     /* batch not in [1, 8]                                */
    QMV_ERR_ALIGN = 6,     /* a pointer is not aligned to its element type        */
    QMV_ERR_OVERFLOW = 7,  /* a size product does not fit the library's limits  */
    QMV_ERR_ALIAS = 8,     /* an output overlaps an input                        */
    QMV_ERR_CUDA = 9,      /* the CUDA runtime reported an error at launch       */
    QMV_ERR_ROW_ID = 10,   /* (device status) a gathered row id was out of range */
    QMV_ERR_ARG = 11       /* a scalar argument (a temperature) is out of range  */
} qmv_status;

/* Largest group the CQ kernels transform (one group must fit in shared
 * memory as float32). */
#define QMV_MAX_GROUP 32768
/* Largest activation batch per call. */
#define QMV_MAX_BATCH 8
/* Largest Hadamard dimension of hadamard_mlp (the vector is transformed
 * in one block's shared memory as float32). */
#define QMV_MAX_HADAMARD 32768

/*
 * A CQ matrix, the page's CqMatrix record ("part 1", section 4): fields
 * output, input, inputPadded, group, bits, rowBytes, packed, norms and the
 * codebook for this bit width.
 *
 *   output        rows (>= 0)
 *   input         logical columns, 1 <= input <= input_padded
 *   input_padded  stored columns P, a multiple of group
 *   group         FWHT group G, a power of two, 2 <= G <= min(P, 32768)
 *   bits          index width b in {2, 3, 4, 5}
 *   row_bytes     must equal ceil(P * b / 8) (the record-length rule of
 *                 "part 1", "Minimal tests")
 *   packed        [output, row_bytes] bytes.  Column k of row r is the
 *                 integer formed by bits [k*b, k*b + b) of the row's
 *                 little-endian bit stream (bit t = byte t/8, bit t%8).  For
 *                 b = 2 this is four codes per byte, low crumb first
 *                 ("part 2", section 3); for b = 4 two codes, low nibble
 *                 first.
 *   norms         [output, P / G] IEEE binary16 bit patterns
 *   codebook      [2^b] float32 levels
 */
typedef struct {
    int64_t output;
    int64_t input;
    int64_t input_padded;
    int64_t group;
    int32_t bits;
    int32_t reserved; /* must be 0 */
    int64_t row_bytes;
    const uint8_t *packed;
    const uint16_t *norms;
    const float *codebook;
} qmv_cq_matrix;

/*
 * cq_prepare -- "part 2", section 2 "Prepare an activation for CQ".
 *
 * For each of `batch` vectors: copy x[v][0..input) into a zero-padded row of
 * input_padded floats, apply the unnormalised FWHT to every group of G
 * consecutive columns (butterfly strides 1, 2, 4, ... in that order, each
 * result rounded to float32, pair (i, i+h) -> (a+b, a-b)), then multiply
 * each element by s = 1/sqrt(G) computed in float64, the product taken in
 * float64 and rounded to float32.  The result is bit-exact to that
 * definition.
 *
 *   m         matrix whose input, input_padded and group are used (its
 *             data pointers are not read and may be NULL)
 *   x         [batch, input] float32
 *   prepared  [batch, input_padded] float32, written
 */
QMV_API qmv_status cq_prepare(const qmv_cq_matrix *m, const float *x, int32_t batch,
                      float *prepared, qmv_stream stream);

/*
 * cq_matvec -- "part 2", section 3 "Dot packed rows directly":
 *
 *   y[v][r] = sum_g f16(norms[r][g]) * sum_{k in group g} codebook[idx(r,k)] * prepared[v][k]
 *
 * accumulated in float32 (fixed order).  Accuracy: within
 * 1e-4 * sum_g |norm| sum_k |codebook * prepared| + 1e-6 of the exact value.
 *
 *   prepared  [batch, input_padded] float32 (normally cq_prepare's output)
 *   y         [batch, output] float32, written
 */
QMV_API qmv_status cq_matvec(const qmv_cq_matrix *m, const float *prepared, int32_t batch,
                     float *y, qmv_stream stream);

/*
 * cq_dequantize_row -- "part 2", "Row gather" (the embedding lookup of
 * section 5).  For each id: per group, every level times the group's norm
 * (one float32 product), the unnormalised FWHT as in cq_prepare, then the
 * 1/sqrt(G) scale as in cq_prepare; the first `input` columns are written.
 * Bit-exact to that definition.
 *
 *   rows        [n] int32 row ids (n >= 0)
 *   out         [n, input] float32, written
 *   dev_status  optional device int32.  An id outside [0, output) gives a
 *               row of zeros and stores QMV_ERR_ROW_ID here (the value is
 *               never reset by the library: the caller zeroes it).
 */
QMV_API qmv_status cq_dequantize_row(const qmv_cq_matrix *m, const int32_t *rows, int64_t n,
                             float *out, int32_t *dev_status, qmv_stream stream);

/* Most matrices one cq_matvec_multi / cq_prepare_matvec call takes. */
#define QMV_MAX_MATRICES 8

/*
 * cq_matvec_multi -- several CQ matrices applied to one prepared activation
 * in one launch.  needle.js "part 2", section 6 ("An optimized backend can
 * reuse the prepared CQ activation for all three": phiPre, phiPost and
 * phiResidual of one normalised input) and section 7 (the Q, K and V
 * projections of one block input).
 *
 * mats[i] for i < nmats (1 <= nmats <= QMV_MAX_MATRICES) must share input,
 * input_padded, group, bits and the codebook array (the archive keeps one
 * codebook per bit width, "part 1" section 4); output, packed and norms are
 * per matrix.  ys[i] (a host array of device pointers) receives matrix i's
 * [batch, output_i] result, exactly what cq_matvec(mats[i], ...) would
 * write.  Every ys[i] must be distinct from every input and every other
 * ys[j] (QMV_ERR_ALIAS); a mismatch of the shared fields is QMV_ERR_SHAPE.
 */
QMV_API qmv_status cq_matvec_multi(const qmv_cq_matrix *mats, int32_t nmats, const float *prepared,
                                   int32_t batch, float *const *ys, qmv_stream stream);

/*
 * cq_prepare_matvec -- cq_prepare fused into cq_matvec_multi: x is
 * prepared ("part 2", section 2) inside the same launch and applied to
 * every matrix.  Results are bitwise equal to cq_prepare followed by
 * cq_matvec_multi.  `prepared` may be NULL; when given, the prepared
 * activation [batch, input_padded] is also written there.  When
 * batch * input_padded floats do not fit on chip (over 96 KiB) or
 * group > 1024, the call runs cq_prepare and cq_matvec_multi as two
 * launches instead (same results; `prepared` must then be given).
 */
QMV_API qmv_status cq_prepare_matvec(const qmv_cq_matrix *mats, int32_t nmats, const float *x,
                                     int32_t batch, float *prepared, float *const *ys,
                                     qmv_stream stream);

/*
 * f8_matvec -- ds4f-disk issue #6, step 1 (the F8 matvec with per-block
 * E8M0 scales; the head of work item 3 has this shape):
 *
 *   y[v][r] = sum_c e4m3(w[r][c]) * e8m0(scale[r*SR/R][c*SC/C]) * x[v][c]
 *
 * with integer floor division.  E4M3: e=0 subnormal m*2^-9, otherwise
 * (1+m/8)*2^(e-7), saturated at 448 (so 0x7F / 0xFF read as +/-448).  E8M0:
 * 2^(e-127); code 255 is NaN.  Accumulated in float32; accuracy within
 * 1e-4 * sum_c |w * s * x| + 1e-6 of the exact value.  At batch 2..8 (C a
 * multiple of 64, C >= 256, 64-column-aligned scale blocks) the products run
 * on the tensor cores: every finite E4M3 value is an f16, and each 64-column
 * block of x is split into f16 parts hi + lo under a power-of-two exponent,
 * which carries an element to 2^-22 of itself or 2^-39 of the block's
 * largest |x|, whichever is larger.  At batch 5..8, when C is a multiple of
 * 128 up to 4096, R is at least 192 rows per SM, every scale block starts on
 * a multiple of 128 columns and of 64 rows, and w and x are 16-byte aligned,
 * the raw E4M3 weights go to the fifth-generation tensor cores instead,
 * against x split per 128-column block into eight E4M3 pieces (an element to
 * 2^-16 of itself or 2^-45 of the block's largest |x|, whichever is larger).
 * That path keeps partial sums in y between two passes over K, so the argmax
 * form without y runs the batch 2..8 kernel above unless its workspace has
 * room for the logits (QMV_F8_ARGMAX_WORKSPACE_TC_BYTES).
 * Non-finite results are recomputed element by element, so NaN and Inf
 * follow the formula above.
 *
 *   w      [R, C] E4M3 bytes, R >= 0, C >= 1
 *   scale  [SR, SC] E8M0 bytes, 1 <= SR <= max(R, 1), 1 <= SC <= C
 *   x      [batch, C] float32
 *   y      [batch, R] float32, written
 */
QMV_API qmv_status f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                     int64_t SR, int64_t SC, const float *x, int32_t batch, float *y,
                     qmv_stream stream);

/*
 * i8_matvec -- ds4f-disk issue #6, step 4: the I8 matvec ("int8 widen,
 * per-16-group E8M0 scales"; step 3's first tokens ran an I8 head):
 *
 *   y[v][r] = sum_c w[r][c] * e8m0(scale[r][c / 16]) * x[v][c]
 *
 * with groups of 16 consecutive columns of a row sharing one E8M0 scale
 * (2^(e-127); code 255 is NaN).  Accumulated in float32; accuracy within
 * 1e-4 * sum_c |w * s * x| + 1e-6 of the exact value.  At batch 1 (C a
 * multiple of 16) each group's products are exact int32 sums over x in
 * fixed point (error at most 2^-30 of the group's largest |x| per element);
 * at batch 2..8 (C a multiple of 64, 256 <= C <= 4096) they run on the
 * tensor cores, with the group scale folded into the f16 weights (exact for
 * scales 2^-24 .. 2^5; rows with other scales are computed element by
 * element) and x split as for f8_matvec.
 *
 *   w      [R, C] int8, R >= 0, C >= 1
 *   scale  [R, ceil(C / 16)] E8M0 bytes
 *   x      [batch, C] float32
 *   y      [batch, R] float32, written
 */
QMV_API qmv_status i8_matvec(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                             const float *x, int32_t batch, float *y, qmv_stream stream);

/*
 * i8_quantize_x -- Mnemonic "In the browser", "Dot products and math": the
 * activations quantized to int8 per group of 32, with one float scale per
 * group, once per vector.  For vector v and group j (columns [32 j, 32 j + 32),
 * the last group shorter when C % 32 != 0):
 *
 *   d[v][j] = m / 127,  m = max |x[v][c]| over the group
 *   q[v][c] = clamp(rint(x[v][c] / d[v][j]), -127, 127)
 *
 * Both divisions are IEEE float32 and rint rounds to nearest even (the page
 * gives no rounding rule; this is the plainest reading), so the codes are
 * exactly those of any IEEE float32 evaluation.  d = 0 (all zeros, or m / 127
 * underflows) gives q = 0; a group holding Inf or NaN gives d = NaN, q = 0.
 *
 *   x       [batch, C] float32, C >= 1
 *   xq      [batch, C] int8, written
 *   xscale  [batch, ceil(C / 32)] float32, written
 * Errors: QMV_ERR_BATCH, QMV_ERR_SHAPE, QMV_ERR_OVERFLOW, QMV_ERR_NULL,
 * QMV_ERR_ALIGN (x or xscale not 4-byte aligned), QMV_ERR_ALIAS, QMV_ERR_CUDA.
 */
QMV_API qmv_status i8_quantize_x(const float *x, int64_t C, int32_t batch, int8_t *xq,
                                 float *xscale, qmv_stream stream);

/*
 * i8_matvec_q8 -- int8 weights times int8 activations, the dot product of
 * Mnemonic "In the browser", "Dot products and math" (exact int32 sums of
 * int8 x int8 products, then floats scaled by the activation group's scale)
 * over the I8 weights of ds4f-disk issue #6, step 4:
 *
 *   y[v][r] = sum_c w[r][c] * e8m0(scale[r][c / 16]) * xq[v][c] * xscale[v][c / 32]
 *
 * Each 16-column group's int8 x int8 sum is exact in int32; the sum times its
 * two scales is accumulated in float32, within 1e-4 * sum_c |w * s * q * d|
 * + 1e-6 of the exact value.  From batch 4 on, matrices large enough to
 * stream (C a multiple of 64, 256 <= C <= 4096) run on the tensor cores
 * instead, with q * d split into f16 hi + lo as i8_matvec splits x (same
 * bound).  xq and xscale are i8_quantize_x's output (any int8 codes and
 * float scales are accepted).
 *
 *   w       [R, C] int8, R >= 0, C >= 1
 *   scale   [R, ceil(C / 16)] E8M0 bytes (code 255 is NaN)
 *   xq      [batch, C] int8
 *   xscale  [batch, ceil(C / 32)] float32
 *   y       [batch, R] float32, written; must not overlap any input
 * Errors: QMV_ERR_BATCH, QMV_ERR_SHAPE, QMV_ERR_OVERFLOW, QMV_ERR_NULL,
 * QMV_ERR_ALIGN (xscale or y not 4-byte aligned), QMV_ERR_ALIAS,
 * QMV_ERR_CUDA.
 */
QMV_API qmv_status i8_matvec_q8(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                                const int8_t *xq, const float *xscale, int32_t batch, float *y,
                                qmv_stream stream);

/*
 * hadamard_mlp -- the Hadamard MLP block of "part 2", section 8, from the
 * normalised block input on.  For each of `batch` vectors:
 *
 *   z = x zero-padded to D values
 *   z[i] = z[i] * d1[i]                      (float32 product)
 *   z = normalizedFwht(z)                    (section-1 butterfly over all D
 *                                             values, strides 1, 2, 4, ...,
 *                                             each result float32, then the
 *                                             float64 product with
 *                                             1/sqrt(D) rounded to float32)
 *   z[i] = silu(d2[i] * z[i])                (silu(v) = v / (1 + e^-v))
 *   z = normalizedFwht(z)
 *   o[i] = z[i] * d3[i]                      for i < n (float32 product)
 *   o[i] = residual[i] + o[i]                if residual is non-NULL
 *   o[i] = o[i] - u[i]                       if u is non-NULL
 *
 * The page's block takes its input from zcrms(afterAttention, weight) and
 * adds afterAttention back before subtracting the lane-mix input u; the
 * pages do not define zcrms, so the caller passes its output as x and
 * afterAttention as residual.  Every step is computed as defined above
 * except silu, which is evaluated in float32 (the page evaluates it in
 * float64): o is within 1e-5 * A of the float64-silu result, A =
 * |d3[i]| / sqrt(D) * sum_j |silu_j| + |residual[i]| + |u[i]|.
 *
 *   x         [batch, n] float32, 1 <= n <= D
 *   D         Hadamard dimension, a power of two, 1 <= D <= QMV_MAX_HADAMARD
 *   d1,d2,d3  [D] float32 diagonals
 *   residual  [batch, n] float32 or NULL
 *   u         [batch, n] float32 or NULL
 *   out       [batch, n] float32, written; must not overlap any input
 * Errors: QMV_ERR_BATCH, QMV_ERR_SHAPE (D not a power of two in range, n
 * outside [1, D]), QMV_ERR_NULL, QMV_ERR_ALIGN (a pointer not 4-byte
 * aligned), QMV_ERR_ALIAS, QMV_ERR_CUDA.
 */
QMV_API qmv_status hadamard_mlp(const float *x, int64_t n, int64_t D, const float *d1,
                                const float *d2, const float *d3, const float *residual,
                                const float *u, int32_t batch, float *out, qmv_stream stream);

/* Bytes of device workspace f8_matvec_argmax needs for `batch` vectors: a
 * 16-byte arrival counter, then one (value, row) partial result per block
 * and vector, for at most QMV_ARGMAX_MAX_BLOCKS blocks. */
#define QMV_ARGMAX_MAX_BLOCKS 2048
#define QMV_ARGMAX_COUNTER_BYTES 16
#define QMV_F8_ARGMAX_WORKSPACE_BYTES(batch) \
    ((int64_t)QMV_ARGMAX_COUNTER_BYTES + (int64_t)QMV_ARGMAX_MAX_BLOCKS * (int64_t)(batch) * 16)
/* Bytes of workspace with which a call without y also keeps its batch x R
 * logits in the workspace (behind the partials, from the next 256-byte
 * boundary), so that batch 5..8 calls can run on the tcgen05 kernel; with less
 * they run on the batch 2..8 kernel. */
#define QMV_F8_ARGMAX_LOGITS_OFFSET(batch) ((QMV_F8_ARGMAX_WORKSPACE_BYTES(batch) + 255) / 256 * 256)
#define QMV_F8_ARGMAX_WORKSPACE_TC_BYTES(batch, R) \
    (QMV_F8_ARGMAX_LOGITS_OFFSET(batch) + (int64_t)(batch) * (int64_t)(R) * 4)

/*
 * f8_matvec_argmax -- the head matvec followed by greedy selection, fused.
 * ds4f-disk issue #6, work item 3 ("logits = head x state" then sampling;
 * the head is the single biggest matvec) and step 3 (head.c: F8_E4M3 +
 * E8M0 head logits and a deterministic sampler); greedy selection is the
 * sampler at temperature zero.
 *
 * Computes y = f8_matvec(w, scale, x) exactly as f8_matvec does, then for
 * each vector v the row index r that maximises y[v][r].  Order: NaN is
 * greater than every number (as numpy/torch argmax); among equal values
 * (and among NaNs) the lowest row wins.  The choice is made on the float32
 * values this call computes, so it is always the argmax of the y this call
 * writes.
 *
 *   y          [batch, R] float32, written when non-NULL (else not stored)
 *   out_index  [batch] int64, written
 *   out_value  [batch] float32, written (y[v][out_index[v]])
 *   workspace  device scratch of workspace_bytes >=
 *              QMV_F8_ARGMAX_WORKSPACE_BYTES(batch), 16-byte aligned,
 *              caller-owned.  Its first QMV_ARGMAX_COUNTER_BYTES bytes are a
 *              counter with which the blocks of a call find the last one to
 *              finish (that block reduces the partial results, so the call is
 *              one launch): fill them with zeros once before the workspace's
 *              first use; every call leaves them zero again.  The rest is
 *              scratch, its contents on entry ignored.  Calls that overlap
 *              on the GPU must not share a workspace.  With y NULL and
 *              workspace_bytes >= QMV_F8_ARGMAX_WORKSPACE_TC_BYTES(batch, R),
 *              the logits are written to the workspace from byte
 *              QMV_F8_ARGMAX_LOGITS_OFFSET(batch) on, as [batch, R] float32,
 *              when that lets a batch 5..8 call run on the tcgen05 kernel
 *              (the results are those of the same call with y given).
 * R >= 1.  Other arguments and errors as f8_matvec.
 */
QMV_API qmv_status f8_matvec_argmax(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                                    int64_t SR, int64_t SC, const float *x, int32_t batch, float *y,
                                    int64_t *out_index, float *out_value, void *workspace,
                                    int64_t workspace_bytes, qmv_stream stream);

/*
 * f8_matvec_argmax_noalloc -- f8_matvec_argmax without a caller workspace.
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory, for example an engine whose
 * memory pool owns the whole device and forbids further cudaMalloc, or a
 * plug-in interface that hands over inputs and outputs but no workspace.
 *
 * Same arguments, results and errors as f8_matvec_argmax, minus the
 * workspace: the scratch is a fixed array of
 * QMV_F8_ARGMAX_WORKSPACE_BYTES(QMV_MAX_BATCH) bytes (256 KiB and 16 bytes)
 * inside the library (one per GPU, held until the process exits), enough
 * for batch <= QMV_MAX_BATCH;
 * anything beyond that returns QMV_ERR_BATCH.  The call allocates nothing.
 * Its first call in each CUDA context (per device, and again after
 * cudaDeviceReset or any other teardown of the device's context) looks up
 * that array's device address with the device current, so make that first
 * call before any stream capture.
 * Every call uses the same array: calls that may run at the same time on the
 * GPU (for example on two streams) race and must be ordered by the caller.
 * The array starts zeroed when the library is loaded, and every call leaves
 * its counter (the first QMV_ARGMAX_COUNTER_BYTES bytes) zero again.
 */
QMV_API qmv_status f8_matvec_argmax_noalloc(const uint8_t *w, int64_t R, int64_t C,
                                            const uint8_t *scale, int64_t SR, int64_t SC,
                                            const float *x, int32_t batch, float *y,
                                            int64_t *out_index, float *out_value,
                                            qmv_stream stream);

/* Largest k of topk_sample and f8_matvec_topk_sample. */
#define QMV_MAX_TOPK 64
/* Most slices the first selection pass makes, over all vectors of a call. */
#define QMV_TOPK_MAX_SLICES 1024
/* Bytes of device workspace topk_sample needs, for any R, batch and k. */
#define QMV_TOPK_WORKSPACE_BYTES ((int64_t)QMV_TOPK_MAX_SLICES * QMV_MAX_TOPK * 8)

/*
 * topk_sample -- top-k temperature sampling over head logits.  ds4f-disk
 * issue #6, work item 3 (the head's logits feed top-k / temperature
 * sampling) and step 3 (the sampler is a softmax driven by a seeded
 * generator, so equal seeds give equal tokens).  The pages give no
 * formulas; for each vector v this call computes:
 *
 *   1. the k best rows of y[v] in the greedy order of f8_matvec_argmax
 *      (NaN above every number, then the larger value, then the lower row;
 *      -0 equals +0), listed best first: rows i_0, ..., i_{k-1}, logits
 *      l_j = y[v][i_j];
 *   2. weights w_j = exp((l_j - l_0) / T) in float32 (so w_0 = 1);
 *   3. cumulative sums c_j = w_0 + ... + w_j and S = c_{k-1}, in float32 by
 *      one fixed-order scan (pairs (w_0, w_1), (w_2, w_3), ... added, then
 *      a scan over the pairs); p_j = w_j / S;
 *   4. the token i_j for the smallest j with c_j > u' * S, where u' is u[v]
 *      clamped into [0, 1] (NaN read as 0); when rounding leaves no such j,
 *      the last j with w_j > 0.
 *
 * Where the formula has no value its limit is used: T = 0 is greedy
 * (token i_0, p = 1, 0, ...); a NaN l_0 gives token i_0 and NaN
 * probabilities; l_0 = +inf shares the weight equally among the +inf
 * entries; when every l_j is -inf the weights are equal.  The rows are
 * exact; weights and probabilities are float32 (exp within a few ulp), so
 * the token is the exact draw except when u' * S falls within rounding of
 * a boundary between two entries.  The random draw is an input: u holds
 * one uniform number per vector, produced by the caller's generator.
 *
 *   y            [batch, R] float32 logits, 1 <= R <= 2^31 - 1
 *   k            1 <= k <= min(R, QMV_MAX_TOPK)
 *   temperature  finite and >= 0, else QMV_ERR_ARG
 *   u            [batch] float32 uniform draws
 *   top_index    [batch, k] int64, written (i_0 .. i_{k-1})
 *   top_value    [batch, k] float32 or NULL (l_0 .. l_{k-1})
 *   top_prob     [batch, k] float32 or NULL (p_0 .. p_{k-1})
 *   token        [batch] int64, written
 *   workspace    device scratch of workspace_bytes >= QMV_TOPK_WORKSPACE_BYTES,
 *                16-byte aligned, caller-owned; contents on entry ignored and
 *                on exit unspecified.  Calls that overlap on the GPU must not
 *                share a workspace.
 * Errors: QMV_ERR_BATCH, QMV_ERR_SHAPE (R or k out of range, workspace too
 * small), QMV_ERR_OVERFLOW (R above 2^31 - 1), QMV_ERR_ARG, QMV_ERR_NULL,
 * QMV_ERR_ALIGN (float pointers 4-byte, int64 8-byte, workspace 16-byte),
 * QMV_ERR_ALIAS (an output or the workspace overlaps an input or another
 * output), QMV_ERR_CUDA.
 */
QMV_API qmv_status topk_sample(const float *y, int64_t R, int32_t batch, int32_t k,
                               float temperature, const float *u, int64_t *top_index,
                               float *top_value, float *top_prob, int64_t *token, void *workspace,
                               int64_t workspace_bytes, qmv_stream stream);

/*
 * f8_matvec_topk_sample -- the head matvec then top-k temperature sampling:
 * y = f8_matvec(w, scale, x) exactly as f8_matvec computes it (y is
 * required and written), then topk_sample(y, ...).  The selection is made
 * on the float32 logits this call writes.  Arguments and errors as the two
 * calls; R >= 1.
 */
QMV_API qmv_status f8_matvec_topk_sample(const uint8_t *w, int64_t R, int64_t C,
                                         const uint8_t *scale, int64_t SR, int64_t SC,
                                         const float *x, int32_t batch, float *y, int32_t k,
                                         float temperature, const float *u, int64_t *top_index,
                                         float *top_value, float *top_prob, int64_t *token,
                                         void *workspace, int64_t workspace_bytes,
                                         qmv_stream stream);

/*
 * i8_matvec_topk_sample -- the I8 head then top-k temperature sampling, the
 * token loop of ds4f-disk issue #6 after step 4 (I8 head over the ~246k
 * vocabulary, then the deterministic sampler): y = i8_matvec(w, scale, x)
 * exactly as i8_matvec computes it (y is required and written), then
 * topk_sample(y, ...).  Arguments and errors as the two calls; R >= 1.
 */
QMV_API qmv_status i8_matvec_topk_sample(const int8_t *w, int64_t R, int64_t C,
                                         const uint8_t *scale, const float *x, int32_t batch,
                                         float *y, int32_t k, float temperature, const float *u,
                                         int64_t *top_index, float *top_value, float *top_prob,
                                         int64_t *token, void *workspace,
                                         int64_t workspace_bytes, qmv_stream stream);

/*
 * qmv_tc_wait_timeouts -- how many waits of the fifth-generation tensor-core
 * F8 kernel (f8_matvec and its argmax / top-k forms at batch 5..8) have run
 * out of their one-second limit on the current device since the library was
 * loaded.  A wait that runs out ends its part of the kernel early and the
 * outputs of that call are not valid.  None is expected; the limit exists so
 * that a fault elsewhere cannot leave the kernel waiting forever.
 *
 *   count  host pointer, written
 *
 * Synchronous: a device-to-host copy on the legacy default stream.
 */
QMV_API qmv_status qmv_tc_wait_timeouts(uint64_t *count);

/* Human-readable name of a status code (static storage). */
QMV_API const char *qmv_status_string(qmv_status status);

/* ABI version of this header: 1. */
QMV_API int32_t qmv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
