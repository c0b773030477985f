// topk_kernels.cu -- top-k temperature sampling over head logits (ds4f-disk
// issue #6, work item 3: the head's logits go to top-k / temperature
// sampling; step 3: a softmax sampler driven by a seeded generator).
//
// Two launches per call.  The first splits every vector's R logits into
// `nb` contiguous slices, one block each, and keeps each slice's k best as
// (order key, row) pairs in the workspace; the second takes the k best of
// those nb * k candidates per vector and draws the token.  When one slice
// covers the whole vector (R <= 4096) the first launch does everything.
//
// Selection inside a block works on order keys (a uint32 that sorts like
// the greedy order: NaN on top, -0 equal to +0) paired with rows.  A
// threshold that at least k entries reach is taken from group maxima, the
// entries reaching it are gathered, and each is ranked by counting the
// gathered entries that beat it (select_tile).  Massive ties fall back to
// an exact radix select: four 8-bit digit passes over the keys, then over
// the complemented rows.  Every result is independent of the slicing, and
// of the order in which threads run.
#include <math.h>

#include "qmv_internal.h"

namespace qmv {
namespace topk {

constexpr int kThreads = 512;
constexpr int kTile = 4096;  // candidates brought on chip per pass
constexpr int kMaxK = QMV_MAX_TOPK;
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kNoRow = 0xffffffffu;  // pads a slice with fewer than k rows
constexpr int kWarps = kThreads / 32;
constexpr int kGroups = kThreads / 4;  // 4-thread groups giving the threshold
constexpr int kCand = 1024;            // most entries ranked directly
constexpr int kE = kTile / kThreads;   // entries per thread and tile

static_assert(kMaxK <= kGroups && kGroups <= kThreads, "tau needs at least k groups");
static_assert(kWarps <= 32, "one warp scans the warp totals");
static_assert(kTile % kThreads == 0 && kCand % kThreads == 0, "loads and ranks per thread");

// Greedy order as a uint32: NaN highest, then larger values, -0 equal to
// +0.  Every logit (including -inf) maps above 0, which marks padding.
__device__ __forceinline__ uint32_t order_key(float f) {
    if (isnan(f)) return 0xffffffffu;
    uint32_t b = __float_as_uint(f);
    if ((b << 1) == 0) b = 0;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The logit behind an order key: the key's inverse, except that keys
// shared by several bit patterns (zero: +0 and -0; NaN: every payload) read
// the logit itself, so values come back bit for bit.
__device__ __forceinline__ float logit_of(uint32_t key, const float *yv, uint32_t row) {
    if (key == 0x80000000u || key == 0xffffffffu) return yv[row];
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

struct Smem {
    uint32_t key[kMaxK + kTile];  // [kMaxK - kept, kMaxK): best so far; then the tile
    uint32_t row[kMaxK + kTile];
    uint64_t cand[kCand];  // gathered entries as composites
    int part[kCand];  // rank of each gathered entry
    uint32_t hist[256];
    uint32_t gmax[kGroups];
    int wsum[kWarps];
    uint32_t digit, need, ties, count, tau;
};

struct Args {
    const float *y;
    int64_t R;
    int k;
    int nb;  // slices (blocks) per vector in the first launch
    float temperature;
    const float *u;
    uint2 *ws;  // [batch][k][nb] (key, row): position j of slice b at [v][j][b]
    int64_t *top_index;
    float *top_value;
    float *top_prob;
    int64_t *token;
};

// Adds the digits of the entries still in the running to the histogram.
// ByRow: entries whose key equals `key_eq`, digits of the complemented row.
template <bool ByRow>
__device__ __forceinline__ void count_digits(Smem &s, int lo, int n, uint32_t key_eq,
                                             uint32_t prefix, uint32_t mask, int shift) {
    const int lane = threadIdx.x & 31;
    for (int b = 0; b < n; b += kThreads) {
        const int i = b + int(threadIdx.x);
        uint32_t d = 0x100u + lane;  // out of the running: a group of its own
        if (i < n) {
            const uint32_t key = s.key[lo + i];
            if (ByRow) {
                const uint32_t r = ~s.row[lo + i];
                if (key == key_eq && (r & mask) == prefix) d = (r >> shift) & 255u;
            } else if ((key & mask) == prefix) {
                d = (key >> shift) & 255u;
            }
        }
        const uint32_t peers = __match_any_sync(kFull, d);
        if (d < 256u && lane == __ffs(peers) - 1) atomicAdd(&s.hist[d], uint32_t(__popc(peers)));
    }
}

// Warp 0: the digit holding the need-th best entry, counting from digit 255
// down; stores it with the count still needed inside it and its size.
__device__ __forceinline__ void find_digit(Smem &s, uint32_t need) {
    const int lane = threadIdx.x & 31;
    uint32_t c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        c[j] = s.hist[8 * lane + j];
        tot += c[j];
    }
    uint32_t incl = tot;  // entries in this lane's bins and every bin above
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(kFull, incl, o);
        if (lane + o < 32) incl += t;
    }
    const uint32_t above = incl - tot;
    if (above < need && need <= incl) {
        uint32_t acc = above;
#pragma unroll
        for (int j = 7; j >= 0; j--) {
            if (acc + c[j] >= need) {
                s.digit = 8 * lane + j;
                s.need = need - acc;
                s.ties = c[j];
                break;
            }
            acc += c[j];
        }
    }
}

// One radix pass: histogram, digit, and the updated prefix.  Returns whether
// the digit's entries are exactly the ones still needed.
template <bool ByRow>
__device__ __forceinline__ bool radix_pass(Smem &s, int lo, int n, uint32_t key_eq, uint32_t &prefix,
                                           uint32_t &mask, uint32_t &need, int shift) {
    if (threadIdx.x < 256) s.hist[threadIdx.x] = 0;
    __syncthreads();
    count_digits<ByRow>(s, lo, n, key_eq, prefix, mask, shift);
    __syncthreads();
    if (threadIdx.x < 32) find_digit(s, need);
    __syncthreads();
    prefix |= s.digit << shift;
    mask |= 0xffu << shift;
    need = s.need;
    return s.ties == need;
}

// Composite order of an entry: larger is better (key, then the lower row).
__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t row) {
    return (uint64_t(key) << 32) | uint32_t(~row);
}

// Radix select of the k best of key/row[lo, lo + n) (n > k) into cand[0, k).
// Used when too many entries reach the threshold for the direct path.
__device__ __noinline__ void radix_select(Smem &s, int lo, int n, int k) {
    uint32_t prefix = 0, mask = 0, need = uint32_t(k);
    bool done = false;
    for (int shift = 24; shift >= 0 && !done; shift -= 8)
        done = radix_pass<false>(s, lo, n, 0, prefix, mask, need, shift);
    // more rows share the k-th best key than are needed: lowest rows first
    uint32_t rprefix = 0, rmask = 0;
    for (int shift = 24; shift >= 0 && !done; shift -= 8)
        done = radix_pass<true>(s, lo, n, prefix, rprefix, rmask, need, shift);
    if (threadIdx.x == 0) s.count = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t key = s.key[lo + i], km = key & mask;
        const bool take = km > prefix || (km == prefix && ((~s.row[lo + i]) & rmask) >= rprefix);
        if (take) {
            const uint32_t slot = atomicAdd(&s.count, 1u);
            if (slot < uint32_t(k)) s.cand[slot] = composite(key, s.row[lo + i]);
        }
    }
}

// Merges one tile of entries, kE per thread in registers (key 0 = no
// entry), into the best-so-far list key/row[kMaxK - kept, kMaxK), keeping
// the best min(k, total) best first.  Returns the new kept.  Every thread
// calls it.
//
// A threshold first: the 4-thread groups' largest keys give 128 group
// maxima, and their k-th largest, tau, has at least k entries at or above
// it (one per group; with k entries kept, the last of them bounds tau from
// below the same way), so every entry below tau is beaten k times and
// drops out.  The entries at or above tau (about k for k = 1, about 90 at
// k = 64 on 4096 spread-out logits) are gathered and each is ranked by
// counting the gathered entries that beat it.  When more than kCand
// entries reach tau (massive ties) an exact radix select takes over.
template <int kE>
__device__ __forceinline__ int select_tile(Smem &s, const uint32_t (&key)[kE], const uint32_t (&row)[kE], int kept,
                          int k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t m = 0;
#pragma unroll
    for (int q = 0; q < kE; q++) m = max(m, key[q]);
    m = max(m, __shfl_xor_sync(kFull, m, 1));
    m = max(m, __shfl_xor_sync(kFull, m, 2));
    if ((lane & 3) == 0) s.gmax[tid >> 2] = m;
    __syncthreads();
    {  // tau = the k-th largest group maximum; 4 threads rank each one
        const int gi = tid >> 2, part = tid & 3;
        const uint32_t a = s.gmax[gi];
        int ra = 0;
#pragma unroll 8
        for (int j = part; j < kGroups; j += 4) {
            const uint32_t g = s.gmax[j];
            ra += (g > a || (g == a && j < gi)) ? 1 : 0;
        }
        ra += __shfl_xor_sync(kFull, ra, 1);
        ra += __shfl_xor_sync(kFull, ra, 2);
        if (part == 0 && ra == k - 1) s.tau = a;
    }
    __syncthreads();
    uint32_t tau = s.tau;
    if (kept == k) tau = max(tau, s.key[kMaxK - 1]);
    tau = max(tau, 1u);  // key 0 marks a missing entry
    const bool kept_in = tid < kept && s.key[kMaxK - kept + tid] >= tau;
    int c = kept_in ? 1 : 0;
#pragma unroll
    for (int q = 0; q < kE; q++) c += (key[q] >= tau) ? 1 : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s.wsum[warp] = incl;
    __syncthreads();
    int base, C;
    {  // every warp scans the warp totals: its exclusive prefix and the sum
        const int wv = lane < kWarps ? s.wsum[lane] : 0;
        int sc = wv;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            const int t = __shfl_up_sync(kFull, sc, o);
            if (lane >= o) sc += t;
        }
        C = __shfl_sync(kFull, sc, kWarps - 1);
        base = __shfl_sync(kFull, sc - wv, warp);
    }
    if (C == 0) return kept;  // a tile of missing entries and nothing kept
    if (C <= kCand) {
        int pos = base + incl - c;
        if (kept_in) s.cand[pos++] = composite(s.key[kMaxK - kept + tid], s.row[kMaxK - kept + tid]);
#pragma unroll
        for (int q = 0; q < kE; q++)
            if (key[q] >= tau) s.cand[pos++] = composite(key[q], row[q]);
    } else {  // every entry to shared memory, behind the kept ones
#pragma unroll
        for (int q = 0; q < kE; q++) {
            s.key[kMaxK + tid + q * kThreads] = key[q];
            s.row[kMaxK + tid + q * kThreads] = row[q];
        }
        __syncthreads();
        radix_select(s, kMaxK - kept, kept + kE * kThreads, k);
        C = k;
    }
    __syncthreads();
    // rank = how many gathered entries beat this one; only ranks below k
    // stay.  The gathered composites are distinct (each row of a vector
    // enters once, and padding, key 0, is never gathered: tau >= 1 on the
    // direct path, and the radix path takes k real entries out of more than
    // kCand), so the ranks are too.  With few entries, `parts` neighbouring
    // lanes split each entry's count.
    int parts = 1;  // a power of two, so a group of lanes adds its parts up
    while (parts < 32 && parts * 2 * C <= kThreads) parts *= 2;
#pragma unroll
    for (int q = 0; q < kCand / kThreads; q++) {
        const int t = tid + q * kThreads, i = t / parts, p = t & (parts - 1);
        int r = 0;
        if (i < C) {
            const uint64_t mine = s.cand[i];
#pragma unroll 4
            for (int j = p; j < C; j += parts) {
                const uint64_t o = s.cand[j];
                r += (o > mine) ? 1 : 0;
            }
        }
        for (int o = 1; o < parts; o <<= 1) r += __shfl_xor_sync(kFull, r, o);
        if (i < C && p == 0) s.part[i] = r;
    }
    const int nkept = C < k ? C : k;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kCand / kThreads; q++) {
        const int i = tid + q * kThreads;
        if (i < C) {
            const int r = s.part[i];
            if (r < nkept) {
                const uint64_t e = s.cand[i];
                s.key[kMaxK - nkept + r] = uint32_t(e >> 32);
                s.row[kMaxK - nkept + r] = ~uint32_t(e);
            }
        }
    }
    __syncthreads();
    return nkept;
}

// Softmax over the k best (sorted in key/row[kMaxK - k, kMaxK)) and the
// draw, by warp 0: lane l holds entries 2l and 2l + 1.  The cumulative sums
// are one fixed-order scan (each lane's pair, then a shuffle scan over the
// lanes); S is the last of them.
__device__ void sample(Smem &s, const Args &a, int v, float uv) {
    if (threadIdx.x >= 32) return;
    const int k = a.k, lane = threadIdx.x, ja = 2 * lane, jb = ja + 1;
    const uint32_t *rows = s.row + (kMaxK - k);
    const float *yv = a.y + int64_t(v) * a.R;
    const float T = a.temperature;
    const uint32_t *keys = s.key + (kMaxK - k);
    const float l0 = logit_of(keys[0], yv, rows[0]);
    const float la = (ja < k) ? logit_of(keys[ja], yv, rows[ja]) : 0.0f;
    const float lb = (jb < k) ? logit_of(keys[jb], yv, rows[jb]) : 0.0f;
    const bool greedy = (T == 0.0f) || isnan(l0);
    auto weight = [&](float l, int j) -> float {
        if (j >= k) return 0.0f;
        if (greedy) return (j == 0) ? 1.0f : 0.0f;
        if (l0 == INFINITY) return (l == INFINITY) ? 1.0f : 0.0f;
        if (l0 == -INFINITY) return 1.0f;
        return expf((l - l0) / T);
    };
    const float wa = weight(la, ja), wb = weight(lb, jb);
    float incl = wa + wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    float excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = 0.0f;
    const float S = __shfl_sync(kFull, incl, 31);
    const float ca = excl + wa, cb = incl;
    const float target = ((uv > 0.0f) ? fminf(uv, 1.0f) : 0.0f) * S;
    const uint32_t above_a = __ballot_sync(kFull, ja < k && ca > target);
    const uint32_t above_b = __ballot_sync(kFull, jb < k && cb > target);
    int pick;
    if (above_a | above_b) {
        const int pa = above_a ? 2 * (__ffs(above_a) - 1) : 2 * kMaxK;
        const int pb = above_b ? 2 * (__ffs(above_b) - 1) + 1 : 2 * kMaxK;
        pick = pa < pb ? pa : pb;
    } else {  // rounding left u' * S at or above every sum: the last nonzero weight
        const uint32_t pos_a = __ballot_sync(kFull, wa > 0.0f), pos_b = __ballot_sync(kFull, wb > 0.0f);
        const int pa = pos_a ? 2 * (31 - __clz(pos_a)) : 0;
        const int pb = pos_b ? 2 * (31 - __clz(pos_b)) + 1 : 0;
        pick = pa > pb ? pa : pb;
    }
    if (lane == 0) a.token[v] = int64_t(rows[pick]);
    const int64_t o = int64_t(v) * k;
    const float qnan = __int_as_float(0x7fc00000);
    if (ja < k) {
        a.top_index[o + ja] = int64_t(rows[ja]);
        if (a.top_value) a.top_value[o + ja] = la;
        if (a.top_prob) a.top_prob[o + ja] = isnan(l0) ? qnan : wa / S;
    }
    if (jb < k) {
        a.top_index[o + jb] = int64_t(rows[jb]);
        if (a.top_value) a.top_value[o + jb] = lb;
        if (a.top_prob) a.top_prob[o + jb] = isnan(l0) ? qnan : wb / S;
    }
}

// FromSlices: candidates are the first launch's (key, row) pairs; otherwise
// logits.  Final: sample from the result; otherwise store it as slice output.
template <bool FromSlices, bool Final>
__global__ void __launch_bounds__(kThreads, 3) topk_kernel(Args a) {
    __shared__ Smem s;
    pdl_wait();
    pdl_trigger();
    const int v = blockIdx.y, k = a.k;
    const float uv = Final ? a.u[v] : 0.0f;  // loaded early; used at the end
    int kept = 0;
    if (!FromSlices) {
        const float *yv = a.y + int64_t(v) * a.R;
        const int64_t tiles = (a.R + kTile - 1) / kTile;
        // slice b = tiles [b * tiles / nb, (b + 1) * tiles / nb)
        const int64_t t0 = int64_t(blockIdx.x) * tiles / a.nb, t1 = int64_t(blockIdx.x + 1) * tiles / a.nb;
        for (int64_t t = t0; t < t1; t++) {
            const int64_t base = t * kTile;
            const int len = int(a.R - base < kTile ? a.R - base : kTile);
            uint32_t key[kE], row[kE];
            float val[kE];
#pragma unroll
            for (int q = 0; q < kE; q++) {
                const int i = int(threadIdx.x) + q * kThreads;
                val[q] = (i < len) ? __ldg(yv + base + i) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < kE; q++) {
                const int i = int(threadIdx.x) + q * kThreads;
                key[q] = (i < len) ? order_key(val[q]) : 0u;
                row[q] = (i < len) ? uint32_t(base + i) : kNoRow;
            }
            kept = select_tile<kE>(s, key, row, kept, k);
        }
    } else {
        // The slices' lists are stored position-major (all slices' best,
        // then all second best, ...): each list is sorted, so this order
        // spreads every slice's best entries over all threads and keeps the
        // group threshold tight, and the reads are contiguous.
        const int n = a.nb * k;  // at most QMV_TOPK_MAX_SLICES * QMV_MAX_TOPK
        const uint2 *src = a.ws + int64_t(v) * n;
        for (int base = 0; base < n; base += kTile) {
            const int len = n - base < kTile ? n - base : kTile;
            uint32_t key[kE], row[kE];
#pragma unroll
            for (int q = 0; q < kE; q++) {
                const int i = int(threadIdx.x) + q * kThreads;
                const uint2 e = (i < len) ? src[base + i] : make_uint2(0u, kNoRow);
                key[q] = e.x;
                row[q] = e.y;
            }
            kept = select_tile<kE>(s, key, row, kept, k);
        }
    }
    if (Final) {
        sample(s, a, v, uv);
    } else if (threadIdx.x < unsigned(k)) {
        const int j = threadIdx.x;
        uint2 e = make_uint2(0u, kNoRow);
        if (j < kept) e = make_uint2(s.key[kMaxK - kept + j], s.row[kMaxK - kept + j]);
        a.ws[(int64_t(v) * k + j) * a.nb + blockIdx.x] = e;
    }
}

}  // namespace topk

int topk_slices(int64_t R, int batch) {
    const int64_t tiles = (R + topk::kTile - 1) / topk::kTile;
    const int64_t cap = QMV_TOPK_MAX_SLICES / batch;
    return int(tiles < cap ? tiles : cap);
}

qmv_status launch_topk_sample(const float *y, int64_t R, int batch, int k, float temperature,
                              const float *u, int64_t *top_index, float *top_value, float *top_prob,
                              int64_t *token, void *workspace, cudaStream_t s) {
    topk::Args a;
    a.y = y;
    a.R = R;
    a.k = k;
    a.nb = topk_slices(R, batch);
    a.temperature = temperature;
    a.u = u;
    a.ws = static_cast<uint2 *>(workspace);
    a.top_index = top_index;
    a.top_value = top_value;
    a.top_prob = top_prob;
    a.token = token;
    const dim3 block(topk::kThreads);
    if (a.nb == 1)
        return from_cuda(launch_pdl(topk::topk_kernel<false, true>, dim3(1, batch), block, 0, s, a));
    cudaError_t e = launch_pdl(topk::topk_kernel<false, false>, dim3(a.nb, batch), block, 0, s, a);
    if (e != cudaSuccess) return QMV_ERR_CUDA;
    return from_cuda(launch_pdl(topk::topk_kernel<true, true>, dim3(1, batch), block, 0, s, a));
}

}  // namespace qmv
