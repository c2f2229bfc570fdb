// common.cuh -- internal definitions shared by the translation units of
// libspecverify.so: workspace records, launch arguments, PTX helpers,
// element unpacking and the fixed-order reductions.  Not a public header.
#pragma once

#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>

#include "spec_verify.h"

namespace specv {

// ------------------------------------------------------------ constants

constexpr int kThreads = 256;            // CTA size of the row and draw kernels
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 4;                // 16-byte vectors in flight per lane
constexpr int kMinSeg = 2048;            // smallest warp segment (elements)
constexpr int kSubW = 1024;              // elements per draw sub-tile (a warp)
constexpr int kHistBins = 2048;          // top-p radix bins per pass (one CTA)
constexpr int kElemCap = 1024;           // top-p select: logits of one histogram bin held in shared memory
constexpr int kNucCap = 1024;            // top-p: nucleus list entries kept per row
constexpr float kToppTry = 9.0f;         // top-p select: first try logits within 9 T of the max
constexpr float kFix = 1099511627776.0f; // 2^40: fixed-point mass unit
constexpr float kNegInf = -INFINITY;

// Row-record flags (the public SPEC_DATA_* bit values).
constexpr uint32_t kFlagNonFinite = SPEC_DATA_ROW_NONFINITE;
constexpr uint32_t kFlagAllNegInf = SPEC_DATA_ROW_ALL_NEG_INF;

// ------------------------------------------------------------ records

struct Partial {       // 16 bytes: one piece of one row
    float m;           // max over the piece
    float s;           // sum of 2^((l - m) c) over the piece (stochastic)
    int32_t arg;       // first index of the max, row-relative (argmax)
    uint32_t flags;
};

struct RowRec {        // 32 bytes: one row, after all its pieces
    float m;           // row max
    float z;           // normaliser over the kept tokens: sum 2^((l - m) c)
    uint32_t lam_key;  // ordered key of the smallest kept logit (0: all kept)
    int32_t arg;       // first argmax (greedy / tree)
    float z_full;      // normaliser over the whole row
    uint32_t flags;    // kFlag* bits
    uint32_t pad[2];
};

struct SeqRec {         // one sequence's accept decision (and debug values)
    int32_t j;         // accepted drafts
    uint32_t bad;      // data-error bits (0: fine)
    float S;           // total weight of the final draw
    uint32_t use_p;    // draw from p_{j+1} (bonus row) instead of the residual
    float pneg, pinv;  // -(m c) and 1/z of the draw's target row
    float qneg, qinv;  // the same for the draft row (residual only)
    uint32_t plam, qlam;  // nucleus keys of the two rows
    uint32_t done;     // the draw is already emitted (top-p nucleus list draw)
    uint32_t pad;
    float P[32];       // p_i(x~_i)
    float Q[32];       // q_i(x~_i)
};

struct Workspace {
    uint32_t *err;         // data-error word
    uint32_t *row_ctr;     // per-row piece arrival counters (self-resetting)
    uint32_t *seq_rows;    // per-sequence finished-row counters (self-resetting)
    uint32_t *seq_ctr;     // per-sequence draw-item arrival counters (self-resetting)
    Partial *partial;      // [rows, pmax]
    RowRec *rows;          // [rows]
    float *sub_sums;       // [B, NS] draw weight of every 1024-element sub-tile
    SeqRec *seqs;          // [B]
    int32_t *nuc_n;        // [B (k+1)] entries of each target row's nucleus list, or -1 (top-p)
    uint4 *nuc;            // [B (k+1), kNucCap] (index, target logit, draft logit at it), index order
    uint32_t *accq;        // acceptance queue: [0] length, [1] CTA arrivals, then [B k] pair ids
    uint32_t *sum;         // [rows, sum_stride] row summaries, one entry per group (top-p / top-k)
    int sum_stride;        // summary entries per row
    uint32_t *defer;       // [rows] 1: the row is left to topp_kernel (reset by it)
    int pmax;              // partial slots per row
};

// Where row r of sequence b lives: rows 0..draft_rows_from-1 of a sequence
// are target rows, the rest are draft rows.
struct RowView {
    const void *target;
    const void *draft;
    int V, R, k;
    int draft_rows_from;   // k+1 (chain) or N (tree)
    int tgt_rows_per_seq;  // k+1 (chain) or N (tree)
};

template <typename T>
__device__ __forceinline__ const T *row_ptr(const RowView &v, int row) {
    const int b = row / v.R, r = row - b * v.R;
    if (r < v.draft_rows_from)
        return static_cast<const T *>(v.target) +
               (static_cast<size_t>(b) * v.tgt_rows_per_seq + r) * v.V;
    return static_cast<const T *>(v.draft) +
           (static_cast<size_t>(b) * v.k + (r - v.draft_rows_from)) * v.V;
}

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two-lane fp32 fused multiply-add and add (round to nearest, each lane
// exactly __fmaf_rn / __fadd_rn): one instruction for two logits.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
        "mov.b64 rc, {%6, %7};\nfma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n.reg .b64 ra, rb, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
        "add.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Atomic add with acquire-release semantics at GPU scope: the calling
// thread's earlier writes are visible to whoever observes the new count,
// and writes released by earlier arrivals are visible to this thread after
// it.  Returns the old value.
__device__ __forceinline__ unsigned arrive(unsigned *ctr, unsigned n) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(ctr), "r"(n) : "memory");
    return old;
}

// Streaming 16-byte load: read-only path, no L1 allocation, 256-byte L2
// prefetch (each logit is read once).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------- element types

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;
    static constexpr uint32_t kNegInfWord = 0xFF800000u;
};
template <> struct Elem<uint16_t> {
    static constexpr int kPerVec = 8;
    static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
};

template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec() {
    return make_uint4(Elem<T>::kNegInfWord, Elem<T>::kNegInfWord, Elem<T>::kNegInfWord,
                      Elem<T>::kNegInfWord);
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4 &q, float (&f)[Elem<T>::kPerVec]);
template <>
__device__ __forceinline__ void unpack<float>(const uint4 &q, float (&f)[4]) {
    f[0] = __uint_as_float(q.x);
    f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z);
    f[3] = __uint_as_float(q.w);
}
template <>
__device__ __forceinline__ void unpack<uint16_t>(const uint4 &q, float (&f)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// NaN-propagating max over a batch of vectors.
template <typename T>
__device__ __forceinline__ float batch_max(const uint4 (&q)[kBatch]);
template <>
__device__ __forceinline__ float batch_max<float>(const uint4 (&q)[kBatch]) {
    float m = kNegInf;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        m = max_nan(m, max_nan(max_nan(__uint_as_float(q[u].x), __uint_as_float(q[u].y)),
                               max_nan(__uint_as_float(q[u].z), __uint_as_float(q[u].w))));
    return m;
}
template <>
__device__ __forceinline__ float batch_max<uint16_t>(const uint4 (&q)[kBatch]) {
    uint32_t m = Elem<uint16_t>::kNegInfWord;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        m = max_nan_bf16x2(m, max_nan_bf16x2(max_nan_bf16x2(q[u].x, q[u].y),
                                             max_nan_bf16x2(q[u].z, q[u].w)));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// NaN-propagating max of one vector.
template <typename T>
__device__ __forceinline__ float batch_max1(const uint4 &q);
template <>
__device__ __forceinline__ float batch_max1<float>(const uint4 &q) {
    return max_nan(max_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                   max_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
}
template <>
__device__ __forceinline__ float batch_max1<uint16_t>(const uint4 &q) {
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(q.x, q.y), max_nan_bf16x2(q.z, q.w));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// Ordered key of a logit: monotone in its value, -0 folded onto +0.  bf16
// values use the top 16 bits (exact: their low 16 bits are zero).
template <typename T>
__device__ __forceinline__ uint32_t okey(float v) {
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0;
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return sizeof(T) == 2 ? (b >> 16) : b;
}

// The float whose okey<float> is k.
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Processed probability of one logit: [key >= lam] 2^(l c - m c) / z, with
// negmc = -(m c) and invz = 1 / z.  Explicit round-to-nearest intrinsics
// keep every call site bitwise identical.
template <typename T>
__device__ __forceinline__ float proc_prob(float l, float c, float negmc, float invz,
                                           uint32_t lam_key) {
    const float e = ex2(__fmaf_rn(l, c, negmc));
    return okey<T>(l) >= lam_key ? __fmul_rn(e, invz) : 0.0f;
}

// ---------------------------------------------------------- combining

__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float c) {
    const float mn = fmaxf(m, m2);
    if (mn == kNegInf) {
        m = mn;
        s = 0.0f;
        return;
    }
    s = __fadd_rn(__fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, mn), c))),
                  __fmul_rn(s2, ex2(__fmul_rn(__fsub_rn(m2, mn), c))));
    m = mn;
}

__device__ __forceinline__ void arg_combine(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

// Butterfly reductions: every lane ends with the same (commutative) result.
__device__ __forceinline__ void warp_reduce_ms(float &m, float &s, uint32_t &fl, float c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
        ms_combine(m, s, m2, s2, c);
    }
}

__device__ __forceinline__ void warp_reduce_arg(float &v, int &i, uint32_t &fl) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
        arg_combine(v, i, v2, i2);
    }
}

// Row flags from the combined max: +inf is non-finite; an all -inf row
// (and no NaN) is flagged as such.
__device__ __forceinline__ uint32_t row_flags(float m, uint32_t fl) {
    if (m == INFINITY) fl |= kFlagNonFinite;
    if (m == kNegInf && !(fl & kFlagNonFinite)) fl |= kFlagAllNegInf;
    return fl;
}

// Split [lo, hi) of a row into a scalar head, 16-byte vectors and a scalar
// tail, by absolute address.
template <typename T>
struct Span {
    int e0, a0, nvec, a1, e1;
    __device__ __forceinline__ Span(const T *rowp, int lo, int hi) : e0(lo), e1(hi) {
        constexpr int P = Elem<T>::kPerVec;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp + lo);
        int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(T));
        if (head > hi - lo) head = hi - lo;
        a0 = lo + head;
        nvec = (hi - a0) / P;
        a1 = a0 + nvec * P;
    }
};

// ------------------------------------------------------ row summaries
//
// A statistics pass over a row also leaves its summary: for every group of
// logits one lane reduced in one batch (kBatch vectors, 32 lanes apart),
// one 32-bit entry: bits 31..16 the group's max, bits 15..2 a bound on the
// max of its other vectors, bits 1..0 the vector holding the max.  Values
// are rounded up to bf16 and stored as 16-bit ordered keys (the bound
// keeps the top 14 bits, rounded up).  A later pass then finds the logits
// above any threshold by reading the summary (one entry per 32 or 16
// logits) and only the vectors that can reach it: mostly one per group.
// A row is split into pieces by the warp segments [w seg, (w+1) seg) of the
// concatenated rows; piece i's groups are stored after those of pieces
// 0..i-1, batch-major (entry b 32 + lane).

constexpr int kGroupVecs = 32 * kBatch;  // vectors per batch of one warp

// Summary entries reserved per row: enough for any segment length >=
// kMinSeg and 4- or 2-byte logits.
__host__ __device__ inline int sum_stride_for(int V) {
    return ((V + 4 * kGroupVecs - 1) / (4 * kGroupVecs) + V / kMinSeg + 3) * 32;
}

// Piece i of row `row` (rows of V logits, segments of seg): [lo, hi).
__device__ __forceinline__ void piece_bounds(int row, int V, long long seg, long long w, int &lo,
                                             int &hi) {
    const long long rbase = static_cast<long long>(row) * V;
    const long long a = w * seg > rbase ? w * seg : rbase;
    const long long b = (w + 1) * seg < rbase + V ? (w + 1) * seg : rbase + V;
    lo = static_cast<int>(a - rbase);
    hi = static_cast<int>(b - rbase);
}

// Summary entries of one piece.
template <typename T>
__device__ __forceinline__ int piece_groups(const T *rowp, int lo, int hi) {
    const Span<T> sp(rowp, lo, hi);
    return (sp.nvec + kGroupVecs - 1) / kGroupVecs * 32;
}

// Summary offset of the piece of `row` in segment w (the sum over the
// row's earlier pieces).
template <typename T>
__device__ __forceinline__ int piece_sum_offset(const T *rowp, int row, int V, long long seg,
                                                long long w) {
    const long long wf = static_cast<long long>(row) * V / seg;
    int off = 0;
    for (long long w2 = wf; w2 < w; ++w2) {
        int lo, hi;
        piece_bounds(row, V, seg, w2, lo, hi);
        off += piece_groups<T>(rowp, lo, hi);
    }
    return off;
}

// Summary key of a value: the 16-bit ordered key of the smallest bf16
// value >= x (x itself for bf16 logits).
__device__ __forceinline__ uint16_t sum_key(float x) {
    uint32_t b = __float_as_uint(x);
    if (!(b & 0x80000000u)) b += 0xFFFFu;  // positive: away from zero (no carry out of bit 31)
    b &= 0xFFFF0000u;                      // negative: toward zero; both round up
    return static_cast<uint16_t>(okey<float>(__uint_as_float(b)) >> 16);
}

// The bf16 value (as float) whose summary key is k.
__device__ __forceinline__ float sum_value(uint32_t k) { return key_float(k << 16); }

// A summary entry from the kBatch vector maxima of one group.
__device__ __forceinline__ uint32_t sum_entry(const float (&mu)[kBatch]) {
    static_assert(kBatch == 4, "two bits name the vector");
    int u1 = 0;
#pragma unroll
    for (int u = 1; u < kBatch; ++u)
        if (!(mu[u] <= mu[u1])) u1 = u;  // the first max (a NaN wins)
    float rest = kNegInf;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        if (u != u1) rest = max_nan(rest, mu[u]);
    const uint32_t k2 = min((static_cast<uint32_t>(sum_key(rest)) + 3u) >> 2, 0x3FFFu);
    return (static_cast<uint32_t>(sum_key(mu[u1])) << 16) | (k2 << 2) | static_cast<uint32_t>(u1);
}
__device__ __forceinline__ float entry_max(uint32_t e) { return sum_value(e >> 16); }
__device__ __forceinline__ float entry_rest(uint32_t e) { return sum_value(e & 0xFFFCu); }
__device__ __forceinline__ int entry_vec(uint32_t e) { return static_cast<int>(e & 3u); }

// Warp scan of one value per lane: exclusive prefix in lane order, and the
// round total defined as (exclusive prefix of lane 31) + (its value).
__device__ __forceinline__ float warp_excl_scan(float v, float &total) {
    const int lane = threadIdx.x & 31;
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl = __fadd_rn(incl, y);
    }
    float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    if (lane == 0) excl = 0.0f;
    total = __shfl_sync(0xFFFFFFFFu, __fadd_rn(excl, v), 31);
    return excl;
}

// ------------------------------------------------- sequence completion

// What the warp that finishes a sequence's last row does with it.
enum SeqWork { kSeqDecide = 0, kSeqGreedy = 1, kSeqNone = 2 };

struct SeqArgs {
    int work;                    // SeqWork
    int list_draw;               // draw from the rows' nucleus lists where they exist (top-p)
    int qprob;                   // the draft rows are fp32 probabilities q, used as given
    const int32_t *draft_tokens; // [B, k]
    const float *uniforms;       // [B, k+1] (kSeqDecide)
    int32_t *out_tokens;         // [B, k+1]
    int32_t *out_num;            // [B]
};

// Weight of nucleus entry e of the draw row (index, target logit, draft
// logit -- or, QP, draft probability -- at that index): p(x), or
// max(0, p(x) - q(x)).
template <typename T, bool QP>
__device__ __forceinline__ float list_weight(uint4 e, float c, bool use_p, float pneg, float pinv,
                                             uint32_t plam, float qneg, float qinv,
                                             uint32_t qlam) {
    const float p = proc_prob<T>(__uint_as_float(e.y), c, pneg, pinv, plam);
    if (use_p) return p;
    const float q = QP ? __uint_as_float(e.z) : proc_prob<T>(__uint_as_float(e.z), c, qneg, qinv, qlam);
    return fmaxf(__fsub_rn(p, q), 0.0f);
}

constexpr int kListRun = 8;  // nucleus-list entries per lane per round (256 per round)

// Weights of one lane's run of kListRun consecutive entries from i0 (zero
// past n); all loads issued before any arithmetic.
template <typename T, bool QP>
__device__ __forceinline__ void list_run(const uint4 *L, int n, int i0, float c, bool use_p,
                                         float pneg, float pinv, uint32_t plam, float qneg,
                                         float qinv, uint32_t qlam, float (&w)[kListRun]) {
    uint4 e[kListRun];
#pragma unroll
    for (int t = 0; t < kListRun; ++t)
        e[t] = i0 + t < n ? __ldcg(L + i0 + t) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int t = 0; t < kListRun; ++t)
        w[t] = i0 + t < n ? list_weight<T, QP>(e[t], c, use_p, pneg, pinv, plam, qneg, qinv, qlam)
                          : 0.0f;
}

// Total weight over a nucleus list: rounds of 32 runs of kListRun entries
// in index order; a run's weights are added in order, the runs of a round
// by warp_excl_scan's association, the rounds in order.
template <typename T, bool QP>
__device__ float list_total(const uint4 *L, int n, float c, bool use_p, float pneg, float pinv,
                            uint32_t plam, float qneg, float qinv, uint32_t qlam) {
    const int lane = threadIdx.x & 31;
    float S = 0.0f;
    for (int r0 = 0; r0 < n; r0 += 32 * kListRun) {
        float w[kListRun];
        list_run<T, QP>(L, n, r0 + lane * kListRun, c, use_p, pneg, pinv, plam, qneg, qinv, qlam,
                        w);
        float v = 0.0f;
#pragma unroll
        for (int t = 0; t < kListRun; ++t) v = __fadd_rn(v, w[t]);
        float rt;
        warp_excl_scan(v, rt);
        S = __fadd_rn(S, rt);
    }
    return S;
}

// The final draw of sequence b from the draw row's nucleus list (top-p):
// every logit outside the target row's nucleus has p = 0, so the residual
// max(0, p - q) and the bonus p both vanish there, and the inverse CDF in
// index order runs over the list alone.  Same rule as the full-row draw:
// the first entry with w > 0 whose cumulative weight exceeds u S (else the
// last with w > 0); an empty residual draws from p instead.  Returns false
// (nothing written) if the row has no list.
template <typename T, bool QP>
__device__ bool list_draw(const RowView &v, const SeqArgs &sa, const Workspace &ws, float c,
                          int b, int j, SeqRec *rec) {
    const int lane = threadIdx.x & 31, k = v.k, R = v.R;
    const int tr = b * (k + 1) + j;  // the draw's target row among the target rows
    const int n = __ldcg(&ws.nuc_n[tr]);
    if (n < 0) return false;
    const RowRec *rr = ws.rows + static_cast<size_t>(b) * R;
    const RowRec *pr = rr + j;
    const RowRec *qr = !QP && j < k ? rr + k + 1 + j : pr;
    const float pneg = -__fmul_rn(__ldcg(&pr->m), c), pinv = __frcp_rn(__ldcg(&pr->z));
    const float qneg = -__fmul_rn(__ldcg(&qr->m), c), qinv = __frcp_rn(__ldcg(&qr->z));
    const uint32_t plam = __ldcg(&pr->lam_key), qlam = __ldcg(&qr->lam_key);
    const uint4 *L = ws.nuc + static_cast<size_t>(tr) * kNucCap;
    bool use_p = j == k;
    float S = list_total<T, QP>(L, n, c, use_p, pneg, pinv, plam, qneg, qinv, qlam);
    if (!(S > 0.0f) && !use_p) {
        use_p = true;
        S = list_total<T, QP>(L, n, c, use_p, pneg, pinv, plam, qneg, qinv, qlam);
    }
    const float target = __fmul_rn(sa.uniforms[static_cast<size_t>(b) * (k + 1) + k], S);
    // The same rounds and association as list_total: the first entry with
    // w > 0 whose cumulative weight exceeds u S, else the last with w > 0.
    float Rsum = 0.0f;
    int pos = -1, lastpos = -1;
    for (int r0 = 0; r0 < n && pos < 0; r0 += 32 * kListRun) {
        const int i0 = r0 + lane * kListRun;
        float w[kListRun];
        list_run<T, QP>(L, n, i0, c, use_p, pneg, pinv, plam, qneg, qinv, qlam, w);
        float rsum = 0.0f;
#pragma unroll
        for (int t = 0; t < kListRun; ++t) rsum = __fadd_rn(rsum, w[t]);
        float rt;
        const float excl = warp_excl_scan(rsum, rt);
        float run = 0.0f;
        int found = -1, lastnz = -1;
#pragma unroll
        for (int t = 0; t < kListRun; ++t) {
            run = __fadd_rn(run, w[t]);
            if (w[t] > 0.0f) {
                lastnz = i0 + t;
                if (found < 0 && __fadd_rn(Rsum, __fadd_rn(excl, run)) > target) found = i0 + t;
            }
        }
        const unsigned hm = __ballot_sync(0xFFFFFFFFu, found >= 0);
        if (hm) pos = __shfl_sync(0xFFFFFFFFu, found, __ffs(hm) - 1);
        const unsigned nz = __ballot_sync(0xFFFFFFFFu, lastnz >= 0);
        if (nz) lastpos = __shfl_sync(0xFFFFFFFFu, lastnz, 31 - __clz(nz));
        Rsum = __fadd_rn(Rsum, rt);
    }
    if (pos < 0) pos = lastpos;
    const int token = pos >= 0 ? static_cast<int>(__ldcg(&L[pos].x)) : -1;
    int32_t *ot = sa.out_tokens + static_cast<size_t>(b) * (k + 1);
    if (lane <= k) {
        int32_t val = -1;
        if (lane < j) val = sa.draft_tokens[static_cast<size_t>(b) * k + lane];
        else if (lane == j) val = token;
        ot[lane] = val;
    }
    if (lane == 0) {
        sa.out_num[b] = j;
        rec->S = S;
        rec->use_p = use_p;
        rec->done = 1u;
    }
    return true;
}

// Accept decisions of sequence b ("3.5 Speculative Decoding", step 3: for
// i = 1..k accept x~_i iff u_i q_i(x~_i) < p_i(x~_i), stop at the first
// rejection).  Lane i tests draft i; ballot + ffs give the first rejection.
// Row records are read through L2 (they were written by other warps).
// Writes the sequence record; a sequence with a data error gets -1 outputs.
// QP: the draft rows are probabilities (q_i(x~_i) is read, not computed,
// and must lie in [0, 1]); the sequence's rows are its k+1 target rows.
template <typename T, bool QP>
__device__ void decide_sequence(const RowView &v, const SeqArgs &sa, const Workspace &ws,
                                float c, int b) {
    const int lane = threadIdx.x & 31, k = v.k, V = v.V, R = v.R;
    const RowRec *rr = ws.rows + static_cast<size_t>(b) * R;
    const T *tgt = static_cast<const T *>(v.target) + static_cast<size_t>(b) * (k + 1) * V;
    const T *drf = static_cast<const T *>(v.draft) + static_cast<size_t>(b) * k * V;
    const float *qpb = static_cast<const float *>(v.draft) + static_cast<size_t>(b) * k * V;
    const float *ub = sa.uniforms + static_cast<size_t>(b) * (k + 1);
    uint32_t bad = 0;
    for (int r = lane; r < R; r += 32) bad |= __ldcg(&rr[r].flags);
    bool accept = true;
    float P = 0.0f, Q = 0.0f;
    if (lane < k) {
        const int x = sa.draft_tokens[static_cast<size_t>(b) * k + lane];
        if (x < 0 || x >= V) {
            bad |= SPEC_DATA_TOKEN_RANGE;
        } else {
            const RowRec *tp = rr + lane;
            P = proc_prob<T>(to_f32(tgt[static_cast<size_t>(lane) * V + x]), c,
                             -__fmul_rn(__ldcg(&tp->m), c), __frcp_rn(__ldcg(&tp->z)),
                             __ldcg(&tp->lam_key));
            if (QP) {
                Q = qpb[static_cast<size_t>(lane) * V + x];
                if (!(Q >= 0.0f && Q <= 1.0f)) bad |= SPEC_DATA_PROB_RANGE;
            } else {
                const RowRec *dq = rr + k + 1 + lane;
                Q = proc_prob<T>(to_f32(drf[static_cast<size_t>(lane) * V + x]), c,
                                 -__fmul_rn(__ldcg(&dq->m), c), __frcp_rn(__ldcg(&dq->z)),
                                 __ldcg(&dq->lam_key));
            }
            accept = __fmul_rn(ub[lane], Q) < P;
        }
    }
    if (lane <= k) {
        const float u = ub[lane];
        if (!(u >= 0.0f && u < 1.0f)) bad |= SPEC_DATA_UNIFORM_RANGE;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, o);
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, lane < k && !accept);
    const int j = rej ? __ffs(rej) - 1 : k;
    SeqRec *rec = ws.seqs + b;
    if (lane < k) {
        rec->P[lane] = P;
        rec->Q[lane] = Q;
    }
    if (lane == 0) {
        // The final draw's rows: target row j and draft row j (residual), or
        // the bonus target row k.
        const RowRec *pr = rr + j;
        const RowRec *qr = !QP && j < k ? rr + k + 1 + j : pr;
        rec->j = j;
        rec->bad = bad;
        rec->S = 0.0f;
        rec->use_p = j == k;
        rec->pneg = -__fmul_rn(__ldcg(&pr->m), c);
        rec->pinv = __frcp_rn(__ldcg(&pr->z));
        rec->plam = __ldcg(&pr->lam_key);
        rec->qneg = -__fmul_rn(__ldcg(&qr->m), c);
        rec->qinv = __frcp_rn(__ldcg(&qr->z));
        rec->qlam = __ldcg(&qr->lam_key);
        rec->done = 0u;
    }
    if (bad) {
        if (lane <= k) sa.out_tokens[static_cast<size_t>(b) * (k + 1) + lane] = -1;
        if (lane == 0) {
            sa.out_num[b] = -1;
            atomicOr(ws.err, bad);
        }
    } else if (sa.list_draw) {
        __syncwarp();
        list_draw<T, QP>(v, sa, ws, c, b, j, rec);
    }
}

// Greedy chain rule ("3.5 Speculative Decoding", end of the proof;
// "Speculative Decoding from First Principles", "Draft, verify, keep what
// matches"): keep drafts while they equal the target's first argmax, then
// emit the argmax of the first mismatching (or the bonus) row.
__device__ __forceinline__ void greedy_sequence(const RowView &v, const SeqArgs &sa,
                                                const Workspace &ws, int b) {
    const int lane = threadIdx.x & 31, k = v.k;
    const RowRec *rr = ws.rows + static_cast<size_t>(b) * (k + 1);
    uint32_t bad = 0;
    int g = -1, x = -1;
    if (lane <= k) {
        bad |= __ldcg(&rr[lane].flags);
        g = __ldcg(&rr[lane].arg);
    }
    if (lane < k) {
        x = sa.draft_tokens[static_cast<size_t>(b) * k + lane];
        if (x < 0 || x >= v.V) bad |= SPEC_DATA_TOKEN_RANGE;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, o);
    const unsigned miss = __ballot_sync(0xFFFFFFFFu, lane < k && x != g);
    const int j = miss ? __ffs(miss) - 1 : k;
    const int gj = __shfl_sync(0xFFFFFFFFu, g, j);
    if (lane <= k) {
        int32_t val = -1;
        if (!bad) val = lane < j ? x : (lane == j ? gj : -1);
        sa.out_tokens[static_cast<size_t>(b) * (k + 1) + lane] = val;
    }
    if (lane == 0) {
        sa.out_num[b] = bad ? -1 : j;
        if (bad) atomicOr(ws.err, bad);
    }
}

// Called by a whole warp right after its lane 0 wrote row `row`'s record:
// counts the row towards its sequence and, for the sequence's last row,
// runs the sequence's completion step.  Returns the sequence whose accept
// decision this warp took (kSeqDecide), else -1.
template <typename T>
__device__ __forceinline__ int row_done(const RowView &v, const SeqArgs &sa,
                                        const Workspace &ws, float c, int row) {
    if (sa.work == kSeqNone) return -1;
    const int lane = threadIdx.x & 31;
    const int b = row / v.R;
    int last = 0;
    if (lane == 0) last = arrive(&ws.seq_rows[b], 1u) == static_cast<unsigned>(v.R - 1);
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    __syncwarp();
    if (!last) return -1;
    if (lane == 0) ws.seq_rows[b] = 0u;
    if (sa.work == kSeqDecide) {
        if (sa.qprob) decide_sequence<T, true>(v, sa, ws, c, b);
        else decide_sequence<T, false>(v, sa, ws, c, b);
        return b;
    }
    greedy_sequence(v, sa, ws, b);
    return -1;
}

// ----------------------------------------------------------- launchers

struct ToppArgs {
    RowView rows;
    SeqArgs seq;
    float c, temperature, top_p;
    int top_k;         // keep the top_k largest logits and their ties first (0: off)
    long long seg;     // warp segment of the statistics grid (the summaries' layout)
    int rows_total;    // rows of the grid
    Workspace ws;
};

struct FinalArgs {
    const void *target;
    const void *draft;     // draft logits (dtype), or fp32 probabilities (qprob)
    int qprob;
    const int32_t *draft_tokens;
    const float *uniforms;
    int B, k, V;
    int NS;            // 1024-element sub-tiles per row
    long long per;     // warps in the final kernel's grid (each takes an even share)
    float c;
    int32_t *out_tokens;
    int32_t *out_num;
    Workspace ws;
};

struct StreamArgs {
    RowView rows;
    SeqArgs seq;
    long long total;   // elements over all rows
    long long seg;     // elements per warp segment
    float c;           // log2(e) / temperature
    Workspace ws;
    FinalArgs fin;     // kind 3: the final draw's arguments
};

struct AcceptArgs {
    RowView rows;      // the verify call's rows (R = 2k+1)
    long long pairs;   // B k (target row i, draft row i) pairs
    long long total;   // pairs * V: the pairs end to end
    long long seg;     // elements per warp segment
    float c;           // log2(e) / temperature
    int list;          // top-p: sum over the target rows' nucleus lists where present
    Workspace ws;
    float *beta;       // [B, k]
    float *tv;         // [B, k] or null
};

struct TreeSampleArgs {
    const void *target;         // [B, N, V]
    const void *draft;          // [B, N, V]
    const int32_t *parents;     // [N]
    const int32_t *node_tokens; // [B, N]
    const float *uniforms;      // [B, N]: 0 the final draw, c node c's test
    int B, N, V, D;
    float c;                    // log2(e) / temperature
    int32_t *out_tokens;
    int32_t *out_num;
    int32_t *out_path;
    Workspace ws;               // row records [B, 2N]: target rows, then draft rows
};

struct TreeMaskArgs {
    const int32_t *parents;  // [B, N]
    const int32_t *pos0;     // [B] or null (0)
    int B, N;
    uint8_t *mask;           // [B, N, N] or null
    float *bias;             // [B, N, N] or null
    int32_t *pos;            // [B, N] or null
    int rows_per_warp;       // 1..32, set by the launcher
};

struct TreeArgs {
    const int32_t *parents;
    const int32_t *node_tokens;
    int B, N, V, D;
    int32_t *out_tokens;
    int32_t *out_num;
    int32_t *out_path;
    Workspace ws;
};

// Resident CTAs of `kernel` (kThreads threads) on the current device,
// cached per device and `slot`; 0 on a CUDA error.  Each kernel has a slot
// of its own: rows.cu 0-3 and 8-9, final.cu 4-7, accept.cu 12-15.
template <typename K>
int resident_ctas(K kernel, int slot, size_t dsmem = 0) {
    constexpr int kMaxDev = 64, kSlots = 16;
    static int cache[kMaxDev][kSlots];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev || slot < 0 ||
        slot >= kSlots)
        return 0;
    int v = __atomic_load_n(&cache[dev][slot], __ATOMIC_RELAXED);
    if (v > 0) return v;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, dsmem) !=
            cudaSuccess)
        return 0;
    v = sms * (per_sm > 0 ? per_sm : 1);
    __atomic_store_n(&cache[dev][slot], v, __ATOMIC_RELAXED);
    return v;
}

// kind 0: stochastic statistics; kind 1: argmax.  dtype: SPEC_F32 /
// SPEC_BF16.  Each returns SPEC_OK or SPEC_ERR_CUDA.
int launch_stream_rows(const RowView &rows, const SeqArgs &seq, int rows_total, float c,
                       const Workspace &ws, int kind, int dtype, cudaStream_t st,
                       const FinalArgs *fin = nullptr, int *drew = nullptr);
// Stochastic statistics plus every row's summary (top-p's first phase);
// *seg gets the warp segment used (the summary's layout depends on it).
int launch_stream_summary(const RowView &rows, int rows_total, float c, const Workspace &ws,
                          int dtype, cudaStream_t st, long long *seg);
// With top-p one CTA per row reduces the row's statistics, selects its
// nucleus and takes the accept decisions (instead of the row kernel).
int launch_topp_rows(const ToppArgs &a, int rows_total, int dtype, cudaStream_t st);
// The per-row select, one warp per row (select.cu); rows it defers are
// taken by topp_kernel.
int launch_select_warp(const ToppArgs &a, int dtype, cudaStream_t st);
// The final kernel is launched as a programmatic dependent of the row kernel.
int launch_final(const FinalArgs &a, int dtype, cudaStream_t st);
int launch_tree(const TreeArgs &a, cudaStream_t st);
// Stochastic tree walk over the row records (treesample.cu).
int launch_tree_sample(const TreeSampleArgs &a, int dtype, cudaStream_t st);
// Tree attention mask / bias / positions for B trees (treemask.cu).
int launch_tree_mask(const TreeMaskArgs &a, cudaStream_t st);
// Acceptance rate per (sequence, position) from a verify call's row records;
// masked: the rows carry nucleus keys (top-p).
int launch_accept(const AcceptArgs &a, int dtype, bool masked, cudaStream_t st);
int launch_intermediates(const Workspace &ws, int B, int k, float *P, float *Q, float *Z,
                         float *S, cudaStream_t st);

}  // namespace specv
