// spec_verify.cu -- sm_103a kernels and C ABI of libspecverify.so, the
// target-side verification step of speculative decoding.
//
// Method (cited by page title and section):
//   "3.5 Speculative Decoding" (llm-learning-path): "The algorithm (one
//   step)", "Proof that the output distribution is exactly p", "Tree
//   verification"; "246 Speculative Decoding" (ai_in_action): 2.2, 3.1, 3.3;
//   "Speculative Decoding: Mathematical Foundations, ..." (llms.blog): "The
//   Modified Rejection Sampling Algorithm"; "Speculative Decoding from First
//   Principles" (theservingstack.com): "Draft, verify, keep what matches".
//
// Data path (one call, all on the caller's stream):
//   rows_kernel   one CTA per (row, tile): streams a tile of one logit row
//                 once from HBM with 16-byte loads and reduces it to a tile
//                 partial (running max + sum of 2^((l - max) * log2(e)/T),
//                 or max + first argmax).  The CTA that finishes a row last
//                 (atomic tile counter, no waiting) combines the row's
//                 partials into the row record and, with top-p on, selects
//                 the nucleus threshold from the row while it is L2-resident.
//   final_kernel  (stochastic) one CTA per (sub-tile, sequence): every CTA
//                 re-derives the sequence's accept decisions from the row
//                 records (warp ballot / ffs over the k positions), then
//                 sums the draw weights of its sub-tile of the residual (or
//                 bonus) row; the CTA that finishes the sequence last picks
//                 the sub-tile holding u * S and scans it for the token.
//   greedy_kernel / tree_kernel  one CTA per sequence: argmax match scan or
//                 the parent-walk of the candidate tree.
//
// Every reduction runs in a fixed order, so a call is bitwise reproducible.
// No kernel waits on another CTA: cross-CTA hand-off uses the "last CTA to
// arrive" pattern only.  Data errors set flags, never trap.

#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>

#include "spec_verify.h"

namespace {

constexpr int kThreads = 256;          // CTA size of the row and draw kernels
constexpr int kWarps = kThreads / 32;
constexpr int kTileMax = 16384;        // elements of a row per rows_kernel CTA
constexpr int kSub = 8192;             // elements per draw sub-tile
constexpr int kRun = kSub / kThreads;  // contiguous elements per thread (32)
constexpr int kBatch = 4;              // 16-byte vectors in flight per thread
constexpr int kHistBins = 2048;        // top-p radix bins per pass
constexpr int kSeqRec = 64;            // floats per sequence debug record
constexpr float kFix = 1099511627776.0f;  // 2^40: fixed-point mass unit
constexpr float kNegInf = -INFINITY;

// Row-record flags (same bit values as the public SPEC_DATA_* bits).
constexpr uint32_t kFlagNonFinite = SPEC_DATA_ROW_NONFINITE;
constexpr uint32_t kFlagAllNegInf = SPEC_DATA_ROW_ALL_NEG_INF;

struct TilePartial {   // 16 bytes
    float m;           // tile max (stochastic) / max value (argmax)
    float s;           // sum of 2^((l - m) c) (stochastic)
    int32_t arg;       // first index of the max (argmax), row-relative
    uint32_t flags;
};

struct RowRec {        // 32 bytes
    float m;           // row max
    float z;           // normaliser over the kept tokens: sum 2^((l - m) c)
    uint32_t lam_key;  // ordered key of the smallest kept logit (0: all)
    int32_t arg;       // first argmax (greedy / tree)
    float z_full;      // normaliser over the whole row
    uint32_t flags;    // kFlag* bits
    uint32_t pad[2];
};

struct Workspace {
    uint32_t *err;         // data-error word
    uint32_t *row_ctr;     // per-row tile arrival counters
    uint32_t *seq_ctr;     // per-sequence sub-tile arrival counters
    TilePartial *partial;  // [rows, T]
    RowRec *rows;          // [rows]
    float *sub_sums;       // [B, S2]
    float *seqrec;         // [B, kSeqRec]
};

// ---------------------------------------------------------------- PTX

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
__device__ __forceinline__ void unpack(const uint4 &q, float (&f)[Elem<T>::kPerVec]);
template <>
__device__ __forceinline__ void unpack<float>(const uint4 &q, float (&f)[4]) {
    f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
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
    for (int u = 0; u < kBatch; ++u) {
        m = max_nan(m, max_nan(max_nan(__uint_as_float(q[u].x), __uint_as_float(q[u].y)),
                               max_nan(__uint_as_float(q[u].z), __uint_as_float(q[u].w))));
    }
    return m;
}
template <>
__device__ __forceinline__ float batch_max<uint16_t>(const uint4 (&q)[kBatch]) {
    uint32_t m = Elem<uint16_t>::kNegInfWord;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        m = max_nan_bf16x2(m, max_nan_bf16x2(max_nan_bf16x2(q[u].x, q[u].y),
                                             max_nan_bf16x2(q[u].z, q[u].w)));
    }
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// Ordered key of a logit: monotone in its value, -0 folded onto +0.  bf16
// values use the top 16 bits (exact, since their low 16 bits are zero).
template <typename T>
__device__ __forceinline__ uint32_t okey(float v) {
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0;
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return sizeof(T) == 2 ? (b >> 16) : b;
}

// Processed probability of one logit: [key >= lam] 2^(l c - m c) / z.
template <typename T>
__device__ __forceinline__ float proc_prob(float l, float c, float negmc, float invz,
                                           uint32_t lam_key) {
    const float e = ex2(__fmaf_rn(l, c, negmc));
    return okey<T>(l) >= lam_key ? __fmul_rn(e, invz) : 0.0f;
}

// ------------------------------------------------------------ reductions

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

// Deterministic block reduction of (m, s, flags); result valid in thread 0.
__device__ void block_reduce_ms(float &m, float &s, uint32_t &fl, float c) {
    __shared__ float sm[kWarps], ss[kWarps];
    __shared__ uint32_t sf[kWarps];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
        ms_combine(m, s, m2, s2, c);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sm[warp] = m;
        ss[warp] = s;
        sf[warp] = fl;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kWarps; ++w) {
            ms_combine(m, s, sm[w], ss[w], c);
            fl |= sf[w];
        }
    }
    __syncthreads();
}

__device__ void block_reduce_arg(float &v, int &i, uint32_t &fl) {
    __shared__ float sv[kWarps];
    __shared__ int si[kWarps];
    __shared__ uint32_t sf[kWarps];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
        arg_combine(v, i, v2, i2);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sv[warp] = v;
        si[warp] = i;
        sf[warp] = fl;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kWarps; ++w) {
            arg_combine(v, i, sv[w], si[w]);
            fl |= sf[w];
        }
    }
    __syncthreads();
}

// Exclusive prefix of v over the CTA's threads in thread order, with the
// total defined as (exclusive prefix of the last thread) + (its v): a
// thread-order running sum ending in the last element reproduces it bit for
// bit.  Fixed association, so bitwise reproducible.
__device__ float block_excl_scan(float v, float &total) {
    __shared__ float wincl[kWarps];
    __shared__ float stotal;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x = __fadd_rn(x, y);
    }
    if (lane == 31) wincl[warp] = x;
    __syncthreads();
    if (warp == 0) {
        float t = lane < kWarps ? wincl[lane] : 0.0f;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o) t = __fadd_rn(t, y);
        }
        __syncwarp();
        if (lane < kWarps) wincl[lane] = t;
    }
    __syncthreads();
    float ex = __shfl_up_sync(0xFFFFFFFFu, x, 1);
    if (lane == 0) ex = 0.0f;
    const float excl = __fadd_rn(warp ? wincl[warp - 1] : 0.0f, ex);
    if (threadIdx.x == kThreads - 1) stotal = __fadd_rn(excl, v);
    __syncthreads();
    total = stotal;
    __syncthreads();
    return excl;
}

// ------------------------------------------------------------- row views

struct RowsArgs {
    const void *target;
    const void *draft;
    int B, k, V;
    int R;        // rows per sequence: 2k+1 (stochastic), k+1 (greedy), N (tree)
    int T, TL;    // tiles per row, tile length (multiple of 8)
    int draft_rows_from;  // first row of a sequence that lives in `draft`
    int tgt_rows_per_seq; // rows of `target` per sequence (k+1 or N)
    float c;      // log2(e) / temperature
    float temperature, top_p;
    int use_topp;
    Workspace ws;
};

template <typename T>
__device__ __forceinline__ const T *row_ptr(const RowsArgs &a, int row) {
    const int b = row / a.R, r = row - b * a.R;
    if (r < a.draft_rows_from)
        return static_cast<const T *>(a.target) +
               (static_cast<size_t>(b) * a.tgt_rows_per_seq + r) * a.V;
    return static_cast<const T *>(a.draft) +
           (static_cast<size_t>(b) * a.k + (r - a.draft_rows_from)) * a.V;
}

// Split [e0, e1) of a row into a scalar head, 16-byte vectors and a scalar
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

// Visit every element of [lo, hi) once, thread-strided (any order).
template <typename T, typename F>
__device__ __forceinline__ void for_each_elem(const T *rowp, int lo, int hi, F &&f) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int tid = threadIdx.x;
    if (tid < sp.a0 - sp.e0) f(to_f32(rowp[sp.e0 + tid]), sp.e0 + tid);
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    for (int v = tid; v < sp.nvec; v += kThreads) {
        float f8[P];
        unpack<T>(__ldg(vp + v), f8);
#pragma unroll
        for (int e = 0; e < P; ++e) f(f8[e], sp.a0 + v * P + e);
    }
    if (tid < sp.e1 - sp.a1) f(to_f32(rowp[sp.a1 + tid]), sp.a1 + tid);
}

// ------------------------------------------------------- tile reductions

// Stochastic tile partial: running max m and s = sum 2^(l c - m c), one
// ex2 per element (the running sum is rescaled once per batch when the max
// grows).
template <typename T>
__device__ __forceinline__ void tile_ms(const T *rowp, int lo, int hi, float c, float &m_run,
                                        float &s_run, uint32_t &fl) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int tid = threadIdx.x;
    auto scalar = [&](float l) {
        if (l != l) {
            fl |= kFlagNonFinite;
            return;
        }
        if (l > m_run) {
            s_run = __fmul_rn(s_run, ex2(__fmul_rn(__fsub_rn(m_run, l), c)));
            m_run = l;
        }
        if (m_run != kNegInf) s_run = __fadd_rn(s_run, ex2(__fmaf_rn(l, c, -__fmul_rn(m_run, c))));
    };
    if (tid < sp.a0 - sp.e0) scalar(to_f32(rowp[sp.e0 + tid]));
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    const uint4 neg = make_uint4(Elem<T>::kNegInfWord, Elem<T>::kNegInfWord,
                                 Elem<T>::kNegInfWord, Elem<T>::kNegInfWord);
    for (int v0 = tid; v0 < sp.nvec; v0 += kThreads * kBatch) {
        uint4 q[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + u * kThreads;
            q[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        }
        const float bm = batch_max<T>(q);
        if (bm != bm) {
            fl |= kFlagNonFinite;
            continue;
        }
        if (bm > m_run) {
            s_run = __fmul_rn(s_run, ex2(__fmul_rn(__fsub_rn(m_run, bm), c)));
            m_run = bm;
        }
        if (m_run == kNegInf) continue;
        const float negmc = -__fmul_rn(m_run, c);
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float f[P];
            unpack<T>(q[u], f);
#pragma unroll
            for (int e = 0; e < P; e += 2) {
                acc0 = __fadd_rn(acc0, ex2(__fmaf_rn(f[e], c, negmc)));
                acc1 = __fadd_rn(acc1, ex2(__fmaf_rn(f[e + 1], c, negmc)));
            }
        }
        s_run = __fadd_rn(s_run, __fadd_rn(acc0, acc1));
    }
    if (tid < sp.e1 - sp.a1) scalar(to_f32(rowp[sp.a1 + tid]));
}

// Argmax tile partial: max value and its first index.
template <typename T>
__device__ __forceinline__ void tile_arg(const T *rowp, int lo, int hi, float &best, int &idx,
                                         uint32_t &fl) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int tid = threadIdx.x;
    auto scalar = [&](float l, int i) {
        if (l != l) fl |= kFlagNonFinite;
        else if (l > best) {
            best = l;
            idx = i;
        }
    };
    if (tid < sp.a0 - sp.e0) scalar(to_f32(rowp[sp.e0 + tid]), sp.e0 + tid);
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    const uint4 neg = make_uint4(Elem<T>::kNegInfWord, Elem<T>::kNegInfWord,
                                 Elem<T>::kNegInfWord, Elem<T>::kNegInfWord);
    for (int v0 = tid; v0 < sp.nvec; v0 += kThreads * kBatch) {
        uint4 q[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + u * kThreads;
            q[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        }
        const float bm = batch_max<T>(q);
        if (bm != bm) {
            fl |= kFlagNonFinite;
            continue;
        }
        if (bm > best) {
            int found = INT_MAX;
#pragma unroll
            for (int u = kBatch - 1; u >= 0; --u) {
                float f[P];
                unpack<T>(q[u], f);
#pragma unroll
                for (int e = P - 1; e >= 0; --e)
                    if (f[e] == bm) found = sp.a0 + (v0 + u * kThreads) * P + e;
            }
            best = bm;
            idx = found;
        }
    }
    if (tid < sp.e1 - sp.a1) scalar(to_f32(rowp[sp.a1 + tid]), sp.a1 + tid);
}

// ------------------------------------------------------------ top-p select

// Nucleus threshold of one row (the kept set is {x : key(l_x) >= lam_key}).
// Reading of the pages (top-p is named, never defined): keep the most
// likely tokens until their mass reaches top_p, all ties of the last one
// kept.  Masses are fixed-point integers (2^-40 units) so every histogram
// sum is exact and order-independent.
//   1. Tokens below c0 = m + T (ln((1 - top_p) Z / V) - ln 2) cannot be in
//      the nucleus: all of them together carry < V e(c0) <= (1 - top_p) Z / 2.
//   2. Histogram the mass of the keys in [klo, khi] into <= 2048 bins (bin 0
//      = highest keys), find the bin where the mass from the top first
//      reaches top_p Z, narrow [klo, khi] to it; repeat until one key.
//      bf16 needs 2 passes, fp32 3; each pass reads the row from L2.
template <typename T>
__device__ void topp_select(const T *rowp, int V, float m, float Z, float c, float temperature,
                            float top_p, uint32_t &lam_key, float &z_kept) {
    __shared__ unsigned long long hist[kHistBins];
    __shared__ unsigned long long s_above, s_kept;
    __shared__ uint32_t s_klo, s_khi;
    __shared__ int s_done;
    __shared__ unsigned long long wsum[kWarps];
    __shared__ int s_cross, s_lastnz;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float negmc = -__fmul_rn(m, c);
    const unsigned long long tgt = __float2ull_rn(__fmul_rn(__fmul_rn(top_p, Z), kFix));
    if (tid == 0) {
        const float c0 = m + temperature * (logf((1.0f - top_p) * Z / static_cast<float>(V)) -
                                            0.69314718f);
        s_klo = okey<T>(fminf(c0, m));
        s_khi = okey<T>(m);
        s_above = 0ull;
        s_kept = tgt;  // replaced by the exact kept mass once a key is chosen
        s_done = 0;
    }
    __syncthreads();
    for (int pass = 0; pass < 4 && !s_done; ++pass) {
        const uint32_t klo = s_klo, khi = s_khi;
        const unsigned long long W = static_cast<unsigned long long>(khi - klo) + 1ull;
        const int nb = W < static_cast<unsigned long long>(kHistBins) ? static_cast<int>(W)
                                                                       : kHistBins;
        for (int i = tid; i < nb; i += kThreads) hist[i] = 0ull;
        __syncthreads();
        for_each_elem<T>(rowp, 0, V, [&](float l, int) {
            const uint32_t key = okey<T>(l);
            if (key < klo || key > khi) return;
            const unsigned long long fx =
                __float2ull_rn(__fmul_rn(ex2(__fmaf_rn(l, c, negmc)), kFix));
            const int bin = static_cast<int>((static_cast<unsigned long long>(khi - key) * nb) / W);
            atomicAdd(&hist[bin], fx);
        });
        __syncthreads();
        // Crossing bin: each thread owns a contiguous chunk of bins.
        const int per = (nb + kThreads - 1) / kThreads;
        const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
        unsigned long long mine = 0ull;
        int lastnz = -1;
        for (int i = b0; i < b1; ++i) {
            mine += hist[i];
            if (hist[i]) lastnz = i;
        }
        unsigned long long x = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        if (tid == 0) {
            s_cross = INT_MAX;
            s_lastnz = -1;
        }
        __syncthreads();
        unsigned long long before = s_above + x - mine;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        {
            unsigned long long run = before;
            for (int i = b0; i < b1; ++i) {
                run += hist[i];
                if (run >= tgt) {
                    atomicMin(&s_cross, i);
                    break;
                }
            }
        }
        if (lastnz >= 0) atomicMax(&s_lastnz, lastnz);
        __syncthreads();
        if (tid == 0) {
            // The range always holds mass (it contains the row max, or a bin
            // chosen for its mass), so b >= 0; clamp regardless.
            const int b = max(0, s_cross != INT_MAX ? s_cross : s_lastnz);
            unsigned long long above = s_above;
            for (int i = 0; i < b; ++i) above += hist[i];
            const unsigned long long lo_off = (static_cast<unsigned long long>(b) * W + nb - 1) / nb;
            const unsigned long long hi_off =
                (static_cast<unsigned long long>(b + 1) * W + nb - 1) / nb - 1;
            s_khi = khi - static_cast<uint32_t>(lo_off);
            s_klo = khi - static_cast<uint32_t>(hi_off);
            s_above = above;
            if (s_khi == s_klo) {
                s_kept = above + hist[b];
                s_done = 1;
            }
        }
        __syncthreads();
    }
    lam_key = s_khi;
    z_kept = __fmul_rn(__ull2float_rn(s_kept), 1.0f / kFix);
    __syncthreads();
}

// -------------------------------------------------------------- kernels

// One CTA per (row, tile).  KIND 0: stochastic stats; KIND 1: argmax.
template <typename T, int KIND, bool TOPP>
__global__ void __launch_bounds__(kThreads, 4) rows_kernel(const RowsArgs a) {
    const int item = blockIdx.x;
    const int row = item / a.T;
    const int tile = item - row * a.T;
    const T *rowp = row_ptr<T>(a, row);
    const int lo = tile * a.TL;
    const int hi = min(a.V, lo + a.TL);
    __shared__ int s_last;

    float m = kNegInf, s = 0.0f;
    int arg = INT_MAX;
    uint32_t fl = 0;
    if (KIND == 0) {
        tile_ms<T>(rowp, lo, hi, a.c, m, s, fl);
        block_reduce_ms(m, s, fl, a.c);
    } else {
        tile_arg<T>(rowp, lo, hi, m, arg, fl);
        block_reduce_arg(m, arg, fl);
    }

    if (a.T > 1) {
        if (threadIdx.x == 0) {
            TilePartial tp;
            tp.m = m;
            tp.s = s;
            tp.arg = arg;
            tp.flags = fl;
            a.ws.partial[item] = tp;
            __threadfence();
            const unsigned prev = atomicAdd(&a.ws.row_ctr[row], 1u);
            s_last = prev == static_cast<unsigned>(a.T - 1);
        }
        __syncthreads();
        if (!s_last) return;
        // Last tile of this row: every other partial is visible.
        __threadfence();
        if (threadIdx.x == 0) a.ws.row_ctr[row] = 0u;
        m = kNegInf;
        s = 0.0f;
        arg = INT_MAX;
        fl = 0;
        if (threadIdx.x < a.T) {
            const TilePartial *pp = a.ws.partial + static_cast<size_t>(row) * a.T + threadIdx.x;
            m = __ldcg(&pp->m);
            s = __ldcg(&pp->s);
            arg = __ldcg(&pp->arg);
            fl = __ldcg(&pp->flags);
        }
        if (KIND == 0) block_reduce_ms(m, s, fl, a.c);
        else block_reduce_arg(m, arg, fl);
    }

    __shared__ float s_m, s_z;
    __shared__ uint32_t s_fl;
    if (threadIdx.x == 0) {
        if (m == INFINITY) fl |= kFlagNonFinite;
        if (m == kNegInf && !(fl & kFlagNonFinite)) fl |= kFlagAllNegInf;
        s_m = m;
        s_z = s;
        s_fl = fl;
    }
    __syncthreads();
    uint32_t lam = 0;
    float zk = s_z;
    if (TOPP && KIND == 0 && s_fl == 0 && a.top_p < 1.0f)
        topp_select<T>(rowp, a.V, s_m, s_z, a.c, a.temperature, a.top_p, lam, zk);
    if (threadIdx.x == 0) {
        RowRec r;
        r.m = s_m;
        r.z = zk;
        r.lam_key = lam;
        r.arg = arg;
        r.z_full = s_z;
        r.flags = s_fl;
        r.pad[0] = r.pad[1] = 0;
        a.ws.rows[row] = r;
    }
}

struct FinalArgs {
    const void *target;
    const void *draft;
    const int32_t *draft_tokens;
    const float *uniforms;
    int B, k, V, S2;
    float c;
    int32_t *out_tokens;
    int32_t *out_num;
    Workspace ws;
};

// Weights of the final draw for the `n` elements of one thread's run
// starting at element x: residual max(0, p - q) or (use_p) p.
template <typename T>
__device__ __forceinline__ void draw_weights(const T *prow, const T *qrow, int x, int n,
                                             bool use_p, const RowRec &pr, const RowRec &qr,
                                             float c, float (&w)[kRun]) {
    const float pneg = -__fmul_rn(pr.m, c), pinv = __frcp_rn(pr.z);
    const float qneg = use_p ? 0.0f : -__fmul_rn(qr.m, c);
    const float qinv = use_p ? 0.0f : __frcp_rn(qr.z);
#pragma unroll
    for (int e = 0; e < kRun; ++e) {
        float wv = 0.0f;
        if (e < n) {
            const float p = proc_prob<T>(to_f32(prow[x + e]), c, pneg, pinv, pr.lam_key);
            if (use_p) {
                wv = p;
            } else {
                const float q = proc_prob<T>(to_f32(qrow[x + e]), c, qneg, qinv, qr.lam_key);
                wv = fmaxf(__fsub_rn(p, q), 0.0f);
            }
        }
        w[e] = wv;
    }
}

template <typename T>
__device__ __forceinline__ float run_sum(const float (&w)[kRun]) {
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < kRun; ++e) s = __fadd_rn(s, w[e]);
    return s;
}

// Stochastic final step.  One CTA per (sequence, sub-tile): blockIdx.x =
// b * S2 + sub.
template <typename T>
__global__ void __launch_bounds__(kThreads) final_kernel(const FinalArgs a) {
    const int b = blockIdx.x / a.S2, sub = blockIdx.x - b * a.S2;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = a.k, V = a.V, R = 2 * k + 1;
    const RowRec *rr = a.ws.rows + static_cast<size_t>(b) * R;
    const T *tgt = static_cast<const T *>(a.target) + static_cast<size_t>(b) * (k + 1) * V;
    const T *drf = static_cast<const T *>(a.draft) + static_cast<size_t>(b) * k * V;

    __shared__ int s_j, s_last, s_tok;
    __shared__ uint32_t s_bad;
    __shared__ float s_P[32], s_Q[32];
    __shared__ float s_sums[SPEC_MAX_V / kSub];
    __shared__ float s_pre[SPEC_MAX_V / kSub];
    __shared__ float s_S, s_t;
    __shared__ int s_sel;

    // 1. Accept decisions of this sequence (identical in every CTA).
    if (warp == 0) {
        uint32_t bad = 0;
        for (int r = lane; r < R; r += 32) bad |= rr[r].flags;
        bool accept = true;
        float P = 0.0f, Q = 0.0f;
        if (lane < k) {
            const int x = a.draft_tokens[static_cast<size_t>(b) * k + lane];
            if (x < 0 || x >= V) {
                bad |= SPEC_DATA_TOKEN_RANGE;
            } else {
                const RowRec tp = rr[lane], dq = rr[k + 1 + lane];
                P = proc_prob<T>(to_f32(tgt[static_cast<size_t>(lane) * V + x]), a.c,
                                 -__fmul_rn(tp.m, a.c), __frcp_rn(tp.z), tp.lam_key);
                Q = proc_prob<T>(to_f32(drf[static_cast<size_t>(lane) * V + x]), a.c,
                                 -__fmul_rn(dq.m, a.c), __frcp_rn(dq.z), dq.lam_key);
                const float u = a.uniforms[static_cast<size_t>(b) * (k + 1) + lane];
                accept = __fmul_rn(u, Q) < P;
            }
        }
        if (lane <= k) {
            const float u = a.uniforms[static_cast<size_t>(b) * (k + 1) + lane];
            if (!(u >= 0.0f && u < 1.0f)) bad |= SPEC_DATA_UNIFORM_RANGE;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, o);
        const unsigned rej = __ballot_sync(0xFFFFFFFFu, lane < k && !accept);
        if (lane == 0) {
            s_j = rej ? __ffs(rej) - 1 : k;
            s_bad = bad;
        }
        s_P[lane] = P;
        s_Q[lane] = Q;
    }
    __syncthreads();
    const uint32_t bad = s_bad;
    if (bad) {
        if (sub == 0) {
            for (int i = tid; i <= k; i += kThreads)
                a.out_tokens[static_cast<size_t>(b) * (k + 1) + i] = -1;
            if (tid == 0) {
                a.out_num[b] = -1;
                atomicOr(a.ws.err, bad);
            }
        }
        return;
    }
    const int j = s_j;
    const bool residual = j < k;
    const T *prow = tgt + static_cast<size_t>(j) * V;
    const T *qrow = residual ? drf + static_cast<size_t>(j) * V : prow;
    const RowRec pr = rr[j];
    const RowRec qr = residual ? rr[k + 1 + j] : pr;

    // 2. This CTA's sub-tile weight total.
    float w[kRun];
    auto subtile_total = [&](int s, bool use_p, float &excl) {
        const int x0 = s * kSub + tid * kRun;
        const int n = max(0, min(kRun, V - x0));
        draw_weights<T>(prow, qrow, x0, n, use_p, pr, qr, a.c, w);
        float total;
        excl = block_excl_scan(run_sum<T>(w), total);
        return total;
    };
    float excl;
    const float mine = subtile_total(sub, !residual, excl);
    if (a.S2 > 1) {
        if (tid == 0) {
            a.ws.sub_sums[static_cast<size_t>(b) * a.S2 + sub] = mine;
            __threadfence();
            const unsigned prev = atomicAdd(&a.ws.seq_ctr[b], 1u);
            s_last = prev == static_cast<unsigned>(a.S2 - 1);
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        if (tid == 0) a.ws.seq_ctr[b] = 0u;
        for (int s = tid; s < a.S2; s += kThreads)
            s_sums[s] = s == sub ? mine : __ldcg(&a.ws.sub_sums[static_cast<size_t>(b) * a.S2 + s]);
    } else if (tid == 0) {
        s_sums[0] = mine;
    }
    __syncthreads();

    // 3. Total weight S and the sub-tile holding u * S.
    bool use_p = !residual;
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 1) + k];
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (warp == 0) {
            const int per = (a.S2 + 31) / 32;
            const int s0 = min(a.S2, lane * per), s1 = min(a.S2, s0 + per);
            float chunk = 0.0f;
            for (int s = s0; s < s1; ++s) chunk = __fadd_rn(chunk, s_sums[s]);
            float x = chunk;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x = __fadd_rn(x, y);
            }
            float run = __shfl_up_sync(0xFFFFFFFFu, x, 1);
            if (lane == 0) run = 0.0f;
            for (int s = s0; s < s1; ++s) {
                s_pre[s] = run;
                run = __fadd_rn(run, s_sums[s]);
            }
            // S: the running total after the last sub-tile.
            const int last_lane = (a.S2 - 1) / per;
            const float S = __shfl_sync(0xFFFFFFFFu, run, last_lane);
            if (lane == 0) {
                s_S = S;
                s_t = __fmul_rn(u, S);
            }
        }
        __syncthreads();
        if (s_S > 0.0f || use_p) break;
        // Residual is zero everywhere: draw from p_{j+1} instead.
        use_p = true;
        for (int s = 0; s < a.S2; ++s) {
            float unused_excl;
            const float t = subtile_total(s, true, unused_excl);
            if (tid == 0) s_sums[s] = t;
        }
        __syncthreads();
    }
    if (warp == 0) {
        const float t = s_t;
        int first = INT_MAX, lastnz = -1;
        for (int s = lane; s < a.S2; s += 32) {
            if (first == INT_MAX && __fadd_rn(s_pre[s], s_sums[s]) > t) first = s;
            if (s_sums[s] > 0.0f) lastnz = s;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
            lastnz = max(lastnz, __shfl_xor_sync(0xFFFFFFFFu, lastnz, o));
        }
        if (lane == 0) s_sel = max(0, first != INT_MAX ? first : lastnz);
    }
    __syncthreads();

    // 4. Scan the chosen sub-tile for the first x with C(x) > u * S.
    const int sel = s_sel;
    const float pre = s_pre[sel], t = s_t;
    float ex_sel;
    subtile_total(sel, use_p, ex_sel);
    int found = INT_MAX, lastpos = -1;
    {
        float run = 0.0f;
        const int x0 = sel * kSub + tid * kRun;
#pragma unroll
        for (int e = 0; e < kRun; ++e) {
            run = __fadd_rn(run, w[e]);
            if (w[e] > 0.0f) {
                lastpos = x0 + e;
                if (found == INT_MAX && __fadd_rn(pre, __fadd_rn(ex_sel, run)) > t) found = x0 + e;
            }
        }
    }
    __shared__ int s_found[kWarps], s_lastpos[kWarps];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        found = min(found, __shfl_xor_sync(0xFFFFFFFFu, found, o));
        lastpos = max(lastpos, __shfl_xor_sync(0xFFFFFFFFu, lastpos, o));
    }
    if (lane == 0) {
        s_found[warp] = found;
        s_lastpos[warp] = lastpos;
    }
    __syncthreads();
    if (tid == 0) {
        int f = INT_MAX, lp = -1;
        for (int i = 0; i < kWarps; ++i) {
            f = min(f, s_found[i]);
            lp = max(lp, s_lastpos[i]);
        }
        s_tok = f != INT_MAX ? f : lp;
    }
    __syncthreads();

    // 5. Emit.
    int32_t *ot = a.out_tokens + static_cast<size_t>(b) * (k + 1);
    for (int i = tid; i <= k; i += kThreads) {
        int32_t v = -1;
        if (i < j) v = a.draft_tokens[static_cast<size_t>(b) * k + i];
        else if (i == j) v = s_tok;
        ot[i] = v;
    }
    if (tid == 0) a.out_num[b] = j;
    float *rec = a.ws.seqrec + static_cast<size_t>(b) * kSeqRec;
    if (tid < k) {
        rec[tid] = s_P[tid];
        rec[k + tid] = s_Q[tid];
    }
    if (tid == 0) rec[2 * k] = s_S;
}

struct GreedyArgs {
    const int32_t *draft_tokens;
    int B, k, V;
    int32_t *out_tokens;
    int32_t *out_num;
    Workspace ws;
};

// Greedy chain: one warp per sequence.
__global__ void __launch_bounds__(32) greedy_kernel(const GreedyArgs a) {
    const int b = blockIdx.x, lane = threadIdx.x, k = a.k;
    const RowRec *rr = a.ws.rows + static_cast<size_t>(b) * (k + 1);
    uint32_t bad = 0;
    int g = -1, x = -1;
    if (lane <= k) {
        const RowRec r = rr[lane];
        bad |= r.flags;
        g = r.arg;
    }
    if (lane < k) {
        x = a.draft_tokens[static_cast<size_t>(b) * k + lane];
        if (x < 0 || x >= a.V) bad |= SPEC_DATA_TOKEN_RANGE;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, o);
    const unsigned miss = __ballot_sync(0xFFFFFFFFu, lane < k && x != g);
    const int j = miss ? __ffs(miss) - 1 : k;
    const int gj = __shfl_sync(0xFFFFFFFFu, g, j);
    if (lane <= k) {
        int32_t v = -1;
        if (!bad) v = lane < j ? x : (lane == j ? gj : -1);
        a.out_tokens[static_cast<size_t>(b) * (k + 1) + lane] = v;
    }
    if (lane == 0) {
        a.out_num[b] = bad ? -1 : j;
        if (bad) atomicOr(a.ws.err, bad);
    }
}

struct TreeArgs {
    const int32_t *parents;
    const int32_t *node_tokens;
    int B, N, V, D;
    int32_t *out_tokens;
    int32_t *out_num;
    int32_t *out_path;
    Workspace ws;
};

constexpr int kTreeThreads = 128;

// Greedy tree: one CTA per sequence.  Node n is accepted iff every edge
// (parent p -> child c) on its root path has token(c) == argmax(p); the
// deepest accepted node wins, ties to the lowest index.
__global__ void __launch_bounds__(kTreeThreads) tree_kernel(const TreeArgs a) {
    const int b = blockIdx.x, tid = threadIdx.x, N = a.N;
    __shared__ int s_par[SPEC_MAX_TREE_NODES], s_g[SPEC_MAX_TREE_NODES], s_tok[SPEC_MAX_TREE_NODES];
    __shared__ uint32_t s_bad;
    __shared__ int s_best;
    if (tid == 0) {
        s_bad = 0;
        s_best = 0;
    }
    __syncthreads();
    uint32_t bad = 0;
    for (int n = tid; n < N; n += kTreeThreads) {
        const int p = a.parents[n];
        if (n == 0 ? p != -1 : (p < 0 || p >= n)) bad |= SPEC_DATA_TREE_SHAPE;
        s_par[n] = p;
        const RowRec r = a.ws.rows[static_cast<size_t>(b) * N + n];
        bad |= r.flags;
        s_g[n] = r.arg;
        const int t = a.node_tokens[static_cast<size_t>(b) * N + n];
        if (n > 0 && (t < 0 || t >= a.V)) bad |= SPEC_DATA_TOKEN_RANGE;
        s_tok[n] = t;
    }
    if (bad) atomicOr(&s_bad, bad);
    __syncthreads();
    int key = 0;  // depth * 2048 + (2047 - n) of the best accepted node
    if (!s_bad) {
        for (int n = tid; n < N; n += kTreeThreads) {
            int depth = 0, c = n;
            bool ok = true;
            while (c != 0) {  // terminates: parents[c] < c
                const int p = s_par[c];
                ok = ok && s_tok[c] == s_g[p];
                c = p;
                ++depth;
            }
            if (depth > a.D) bad |= SPEC_DATA_TREE_SHAPE;
            if (ok) key = max(key, depth * 2048 + (2047 - n));
        }
        if (bad) atomicOr(&s_bad, bad);
        atomicMax(&s_best, key);
    }
    __syncthreads();
    const int W = a.D + 1;
    int32_t *ot = a.out_tokens + static_cast<size_t>(b) * W;
    int32_t *op = a.out_path ? a.out_path + static_cast<size_t>(b) * W : nullptr;
    if (s_bad) {
        for (int i = tid; i < W; i += kTreeThreads) {
            ot[i] = -1;
            if (op) op[i] = -1;
        }
        if (tid == 0) {
            a.out_num[b] = -1;
            atomicOr(a.ws.err, s_bad);
        }
        return;
    }
    const int best = 2047 - (s_best & 2047), d = s_best >> 11;
    for (int i = tid; i < W; i += kTreeThreads) {
        if (i > d) {
            ot[i] = -1;
            if (op) op[i] = -1;
        }
    }
    if (tid == 0) {
        int c = best;
        for (int i = d; i >= 0; --i) {
            if (op) op[i] = c;
            if (i > 0) ot[i - 1] = s_tok[c];
            c = s_par[c];
        }
        ot[d] = s_g[best];
        a.out_num[b] = d;
    }
}

__global__ void intermediates_kernel(const Workspace ws, int B, int k, float *P, float *Q,
                                     float *Z, float *S) {
    const int b = blockIdx.x, t = threadIdx.x, R = 2 * k + 1;
    const float *rec = ws.seqrec + static_cast<size_t>(b) * kSeqRec;
    if (t < k) {
        if (P) P[static_cast<size_t>(b) * k + t] = rec[t];
        if (Q) Q[static_cast<size_t>(b) * k + t] = rec[k + t];
    }
    if (Z)
        for (int r = t; r < R; r += blockDim.x)
            Z[static_cast<size_t>(b) * R + r] = ws.rows[static_cast<size_t>(b) * R + r].z;
    if (S && t == 0) S[b] = rec[2 * k];
}

// ------------------------------------------------------------ host side

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int tiles_for(int V) { return (V + kTileMax - 1) / kTileMax; }
int tile_len(int V, int T) { return ((V + T - 1) / T + 7) / 8 * 8; }
int subs_for(int V) { return (V + kSub - 1) / kSub; }

// Carve the workspace; returns the bytes needed (ws may be null).
size_t carve(void *base, int B, int rows_per_seq, int V, Workspace *ws) {
    const size_t rows = static_cast<size_t>(B) * rows_per_seq;
    const int T = tiles_for(V), S2 = subs_for(V);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return static_cast<char *>(base) + o;
    };
    char *err = take(kAlign);
    char *row_ctr = take(rows * sizeof(uint32_t));
    char *seq_ctr = take(static_cast<size_t>(B) * sizeof(uint32_t));
    char *partial = take(rows * T * sizeof(TilePartial));
    char *rowrec = take(rows * sizeof(RowRec));
    char *subs = take(static_cast<size_t>(B) * S2 * sizeof(float));
    char *seqrec = take(static_cast<size_t>(B) * kSeqRec * sizeof(float));
    if (ws) {
        ws->err = reinterpret_cast<uint32_t *>(err);
        ws->row_ctr = reinterpret_cast<uint32_t *>(row_ctr);
        ws->seq_ctr = reinterpret_cast<uint32_t *>(seq_ctr);
        ws->partial = reinterpret_cast<TilePartial *>(partial);
        ws->rows = reinterpret_cast<RowRec *>(rowrec);
        ws->sub_sums = reinterpret_cast<float *>(subs);
        ws->seqrec = reinterpret_cast<float *>(seqrec);
    }
    return off;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int chain_sizes_ok(int B, int k, int V) {
    if (B < 0 || k < 1 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return 0;
    const long long items = static_cast<long long>(B) * (2 * k + 1) * tiles_for(V);
    const long long draws = static_cast<long long>(B) * subs_for(V);
    return items < INT_MAX && draws < INT_MAX;
}

int launch_status() {
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
int launch_rows(const RowsArgs &a, int kind, int rows_total, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>(rows_total) * a.T;
    if (kind == 1) rows_kernel<T, 1, false><<<grid, kThreads, 0, st>>>(a);
    else if (a.use_topp) rows_kernel<T, 0, true><<<grid, kThreads, 0, st>>>(a);
    else rows_kernel<T, 0, false><<<grid, kThreads, 0, st>>>(a);
    return launch_status();
}


struct ChainPlan {
    RowsArgs rows;
    FinalArgs fin;
    GreedyArgs greedy;
    int stoch, dtype, rows_total;
    cudaStream_t st;
};

int plan_chain(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
               const float *uniforms, int B, int k, int V, float temperature, float top_p,
               int mode, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
               void *workspace, size_t workspace_bytes, spec_stream_t stream, ChainPlan *plan) {
    if (mode != SPEC_STOCHASTIC && mode != SPEC_GREEDY) return SPEC_ERR_MODE;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    const bool stoch = mode == SPEC_STOCHASTIC;
    if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted || !workspace)
        return SPEC_ERR_NULL;
    if (stoch && (!draft_logits || !uniforms)) return SPEC_ERR_NULL;
    if (stoch && (!(temperature > 0.0f) || !std::isfinite(temperature) || !(top_p > 0.0f) ||
                  !(top_p <= 1.0f)))
        return SPEC_ERR_PARAM;
    const size_t esz = dtype == SPEC_F32 ? 4 : 2;
    if (!aligned(target_logits, esz) || (stoch && !aligned(draft_logits, esz)) ||
        !aligned(draft_tokens, 4) || (stoch && !aligned(uniforms, 4)) ||
        !aligned(out_tokens, 4) || !aligned(out_num_accepted, 4) || !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < carve(nullptr, B, 2 * k + 1, V, nullptr)) return SPEC_ERR_WORKSPACE;

    RowsArgs &ra = plan->rows;
    ra = RowsArgs{};
    ra.target = target_logits;
    ra.draft = draft_logits;
    ra.B = B;
    ra.k = k;
    ra.V = V;
    ra.R = stoch ? 2 * k + 1 : k + 1;
    ra.T = tiles_for(V);
    ra.TL = tile_len(V, ra.T);
    ra.draft_rows_from = k + 1;
    ra.tgt_rows_per_seq = k + 1;
    ra.temperature = stoch ? temperature : 1.0f;
    ra.c = static_cast<float>(1.4426950408889634 / static_cast<double>(ra.temperature));
    ra.top_p = stoch ? top_p : 1.0f;
    ra.use_topp = stoch && top_p < 1.0f;
    carve(workspace, B, 2 * k + 1, V, &ra.ws);

    FinalArgs &fa = plan->fin;
    fa = FinalArgs{};
    fa.target = target_logits;
    fa.draft = draft_logits;
    fa.draft_tokens = draft_tokens;
    fa.uniforms = uniforms;
    fa.B = B;
    fa.k = k;
    fa.V = V;
    fa.S2 = subs_for(V);
    fa.c = ra.c;
    fa.out_tokens = out_tokens;
    fa.out_num = out_num_accepted;
    fa.ws = ra.ws;

    GreedyArgs &ga = plan->greedy;
    ga = GreedyArgs{};
    ga.draft_tokens = draft_tokens;
    ga.B = B;
    ga.k = k;
    ga.V = V;
    ga.out_tokens = out_tokens;
    ga.out_num = out_num_accepted;
    ga.ws = ra.ws;

    plan->stoch = stoch;
    plan->dtype = dtype;
    plan->rows_total = B * ra.R;
    plan->st = reinterpret_cast<cudaStream_t>(stream);
    return SPEC_OK;
}

int launch_chain_rows(const ChainPlan &p) {
    return p.dtype == SPEC_F32 ? launch_rows<float>(p.rows, p.stoch ? 0 : 1, p.rows_total, p.st)
                               : launch_rows<uint16_t>(p.rows, p.stoch ? 0 : 1, p.rows_total, p.st);
}

int launch_chain_finish(const ChainPlan &p) {
    if (p.stoch) {
        const unsigned grid = static_cast<unsigned>(p.fin.B) * p.fin.S2;
        if (p.dtype == SPEC_F32) final_kernel<float><<<grid, kThreads, 0, p.st>>>(p.fin);
        else final_kernel<uint16_t><<<grid, kThreads, 0, p.st>>>(p.fin);
    } else {
        greedy_kernel<<<p.greedy.B, 32, 0, p.st>>>(p.greedy);
    }
    return launch_status();
}

}  // namespace

extern "C" {

int spec_verify_workspace_size(int B, int k, int V, size_t *bytes) {
    if (!bytes) return SPEC_ERR_NULL;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    *bytes = carve(nullptr, B, 2 * k + 1, V, nullptr);
    return SPEC_OK;
}

int spec_verify_tree_workspace_size(int B, int N, int V, size_t *bytes) {
    if (!bytes) return SPEC_ERR_NULL;
    if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V)
        return SPEC_ERR_SHAPE;
    if (static_cast<long long>(B) * N * tiles_for(V) >= INT_MAX) return SPEC_ERR_SHAPE;
    *bytes = carve(nullptr, B, N, V, nullptr);
    return SPEC_OK;
}

int spec_verify_workspace_init(void *workspace, size_t bytes, spec_stream_t stream) {
    if (!workspace) return SPEC_ERR_NULL;
    return cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
}

int spec_verify_sample(const void *target_logits, const void *draft_logits,
                       const int32_t *draft_tokens, const float *uniforms, int B, int k, int V,
                       float temperature, float top_p, int mode, int dtype,
                       int32_t *out_tokens, int32_t *out_num_accepted, void *workspace,
                       size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V, temperature,
                        top_p, mode, dtype, out_tokens, out_num_accepted, workspace,
                        workspace_bytes, stream, &plan);
    if (rc != SPEC_OK || B == 0) return rc;
    rc = launch_chain_rows(plan);
    if (rc != SPEC_OK) return rc;
    return launch_chain_finish(plan);
}

int spec_verify_sample_rows(const void *target_logits, const void *draft_logits,
                            const int32_t *draft_tokens, const float *uniforms, int B, int k,
                            int V, float temperature, float top_p, int mode, int dtype,
                            int32_t *out_tokens, int32_t *out_num_accepted, void *workspace,
                            size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    const int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V,
                              temperature, top_p, mode, dtype, out_tokens, out_num_accepted,
                              workspace, workspace_bytes, stream, &plan);
    if (rc != SPEC_OK || B == 0) return rc;
    return launch_chain_rows(plan);
}

int spec_verify_sample_finish(const void *target_logits, const void *draft_logits,
                              const int32_t *draft_tokens, const float *uniforms, int B, int k,
                              int V, float temperature, float top_p, int mode, int dtype,
                              int32_t *out_tokens, int32_t *out_num_accepted, void *workspace,
                              size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    const int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V,
                              temperature, top_p, mode, dtype, out_tokens, out_num_accepted,
                              workspace, workspace_bytes, stream, &plan);
    if (rc != SPEC_OK || B == 0) return rc;
    return launch_chain_finish(plan);
}

int spec_verify_tree(const void *target_logits, const int32_t *parents,
                     const int32_t *node_tokens, int B, int N, int V, int D, int dtype,
                     int32_t *out_tokens, int32_t *out_num_accepted, int32_t *out_path,
                     void *workspace, size_t workspace_bytes, spec_stream_t stream) {
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
    if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V || D < 0 || D >= N)
        return SPEC_ERR_SHAPE;
    if (static_cast<long long>(B) * N * tiles_for(V) >= INT_MAX) return SPEC_ERR_SHAPE;
    if (!target_logits || !parents || !node_tokens || !out_tokens || !out_num_accepted ||
        !workspace)
        return SPEC_ERR_NULL;
    const size_t esz = dtype == SPEC_F32 ? 4 : 2;
    if (!aligned(target_logits, esz) || !aligned(parents, 4) || !aligned(node_tokens, 4) ||
        !aligned(out_tokens, 4) || !aligned(out_num_accepted, 4) ||
        (out_path && !aligned(out_path, 4)) || !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < carve(nullptr, B, N, V, nullptr)) return SPEC_ERR_WORKSPACE;
    if (B == 0) return SPEC_OK;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    RowsArgs ra{};
    ra.target = target_logits;
    ra.draft = nullptr;
    ra.B = B;
    ra.k = 0;
    ra.V = V;
    ra.R = N;
    ra.T = tiles_for(V);
    ra.TL = tile_len(V, ra.T);
    ra.draft_rows_from = N;
    ra.tgt_rows_per_seq = N;
    ra.temperature = 1.0f;
    ra.c = 1.4426950408889634f;
    ra.top_p = 1.0f;
    carve(workspace, B, N, V, &ra.ws);
    int rc = dtype == SPEC_F32 ? launch_rows<float>(ra, 1, B * N, st)
                               : launch_rows<uint16_t>(ra, 1, B * N, st);
    if (rc != SPEC_OK) return rc;
    TreeArgs ta{};
    ta.parents = parents;
    ta.node_tokens = node_tokens;
    ta.B = B;
    ta.N = N;
    ta.V = V;
    ta.D = D;
    ta.out_tokens = out_tokens;
    ta.out_num = out_num_accepted;
    ta.out_path = out_path;
    ta.ws = ra.ws;
    tree_kernel<<<B, kTreeThreads, 0, st>>>(ta);
    return launch_status();
}

int spec_verify_last_error(void *workspace, size_t workspace_bytes, spec_stream_t stream) {
    if (!workspace) return SPEC_ERR_NULL;
    if (workspace_bytes < sizeof(uint32_t)) return SPEC_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof word, st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_CUDA;
    return static_cast<int>(word);
}

int spec_verify_intermediates(const void *workspace, size_t workspace_bytes, int B, int k, int V,
                              float *P, float *Q, float *Z, float *S, spec_stream_t stream) {
    if (!workspace) return SPEC_ERR_NULL;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    if (workspace_bytes < carve(nullptr, B, 2 * k + 1, V, nullptr)) return SPEC_ERR_WORKSPACE;
    if (B == 0) return SPEC_OK;
    Workspace ws;
    carve(const_cast<void *>(workspace), B, 2 * k + 1, V, &ws);
    intermediates_kernel<<<B, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ws, B, k, P, Q, Z,
                                                                               S);
    return launch_status();
}

const char *spec_verify_status_string(int status) {
    switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_NULL: return "a required pointer is NULL";
    case SPEC_ERR_SHAPE: return "a size argument is outside the supported range";
    case SPEC_ERR_PARAM: return "temperature must be finite and > 0, top_p in (0, 1]";
    case SPEC_ERR_DTYPE: return "dtype must be SPEC_F32 or SPEC_BF16";
    case SPEC_ERR_MODE: return "mode must be SPEC_STOCHASTIC or SPEC_GREEDY";
    case SPEC_ERR_ALIGN: return "a pointer is misaligned for its element type";
    case SPEC_ERR_WORKSPACE: return "workspace is NULL or too small";
    case SPEC_ERR_CUDA: return "a CUDA runtime call failed";
    case SPEC_DATA_ROW_NONFINITE: return "a logit row holds NaN or +inf";
    case SPEC_DATA_ROW_ALL_NEG_INF: return "a logit row is entirely -inf";
    case SPEC_DATA_TOKEN_RANGE: return "a token lies outside [0, V)";
    case SPEC_DATA_UNIFORM_RANGE: return "a uniform lies outside [0, 1)";
    case SPEC_DATA_TREE_SHAPE: return "parents is not a rooted tree in topological order "
                                      "within depth D";
    default: return "unknown status";
    }
}

}  // extern "C"
