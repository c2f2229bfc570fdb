// topp.cu -- the top-p (nucleus) threshold of every row, and the accept
// decisions that depend on it.
//
// "3.5 Speculative Decoding" (llm-learning-path), "Notation": p and q are
// the target and draft distributions after temperature and top-p; the
// pages name the nucleus but never define it.  Reading: keep the most
// likely tokens until their mass reaches top_p, all ties of the last one
// kept; the kept set is {x : key(l_x) >= lam}, lam the largest key whose
// mass from the top reaches top_p Z.  Masses are fixed-point integers
// (2^-40 units) so every histogram sum is exact and order-independent.
//
// topp_kernel, one CTA per row:
//   1. Statistics and the list.  Fused (top-p alone, the call's first
//      kernel): the CTA streams its row -- max m, normaliser Z, and per
//      warp the summary of its piece in shared memory (the max of every
//      group of logits one lane reduces in one batch) -- then reads again
//      the groups within kToppTry T of m (a nucleus usually ends above
//      m - kToppTry T) into a shared list; rows too long for the shared
//      summary keep instead the logits near the running max as they
//      stream by.  Not fused (top-k: rows the warp select of select.cu
//      deferred): m, Z and the summary come from the statistics grid
//      (rows.cu, kind 2), and the list is every logit >= a lower bound of
//      the K-th largest (the K-th largest group max).
//   2. Tokens below c0 = m + T (ln((1 - top_p) Z / V) - ln 2) cannot be in
//      the nucleus: all of them together carry < V e(c0) <= (1 - top_p) Z / 2.
//   3. Pass A histograms the mass of the listed logits >= y by value,
//      uniformly over [y, m] (bins of keys would crowd the bulk of a row
//      into a few bins: keys are log-spaced), y = max(c0, m - kToppTry T);
//      if that mass falls short of top_p Z it runs again with y = c0, from
//      the row.  The bin where the mass from the top first reaches top_p Z
//      holds lam.
//   4. Pass B gathers the logits of that bin -- the same float arithmetic
//      decides membership in both passes -- and histograms them by key,
//      narrowing until one key is left: the largest key whose mass from the
//      top reaches top_p Z.  (A bin holding more than kElemCap logits is
//      narrowed from the row.)
//   The row record gets lam and the kept mass; the warp that finishes a
//   sequence's last row takes its accept decision.
//   With top-k (a processor the target and the draft must share, "246
//   Speculative Decoding", 6) the same select first runs by count: the
//   K-th largest key, ties kept; top-p then runs on the kept set, its
//   target top_p times the kept set's mass.

#include "stream.cuh"

namespace specv {
namespace {

constexpr int kTpThreads = 256;  // one CTA per row
constexpr int kTpWarps = kTpThreads / 32;
constexpr int kAList = 3072;     // gathered logits held in shared memory
// Shared memory requested per fused CTA: more than the select needs, so that
// at most three CTAs share an SM and the rows being selected (3 x 152 rows
// of ~256 KB for bf16 V=128k) mostly stay in the 126 MB L2 between a CTA's
// two reads of its row.  (Measured on c4: 2 per SM leaves HBM idle while
// both CTAs of an SM select; 4 per SM spills registers and overflows L2;
// 6 CTAs of 128 threads per SM, one wave, takes 1.7x as long.)
constexpr int kToppSmem = 72 * 1024;

struct SelShared {
    unsigned long long hist[kHistBins];
    unsigned long long wsum[kTpWarps];
    unsigned long long b_above, hb;
    int cross, lastnz;
};

// Block-wide scan of the histogram and the crossing bin: the first bin
// (from the top) where above + the mass so far reaches tgt, else the last
// bin holding mass (or 0).  Returns the bin; *b_above gets the mass of the
// bins before it, *hb the bin's own mass, *crossed whether it crossed.
__device__ int cta_cross(SelShared &sh, int nb, unsigned long long above, unsigned long long tgt,
                         unsigned long long *b_above, unsigned long long *hb, bool *crossed) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kPer = kHistBins / kTpThreads;
    unsigned long long h[kPer], mine = 0ull;
    int lastnz = -1;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        h[i] = sh.hist[tid * kPer + i];
        mine += h[i];
        if (h[i]) lastnz = tid * kPer + i;
    }
    unsigned long long x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.wsum[warp] = x;
    __syncthreads();
    unsigned long long before = above + x - mine;
    for (int i = 0; i < warp; ++i) before += sh.wsum[i];
    {
        unsigned long long run = before;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            run += h[i];
            if (run >= tgt && tid * kPer + i < nb) {
                atomicMin(&sh.cross, tid * kPer + i);
                break;
            }
        }
    }
    if (lastnz >= 0) atomicMax(&sh.lastnz, lastnz);
    __syncthreads();
    *crossed = sh.cross != INT_MAX;
    const int b = *crossed ? sh.cross : max(sh.lastnz, 0);
    if (tid == b / kPer) {
        unsigned long long run = before;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if (tid * kPer + i < b) run += h[i];
        sh.b_above = run;
        sh.hb = h[b - tid * kPer];
    }
    __syncthreads();
    *b_above = sh.b_above;
    *hb = sh.hb;
    __syncthreads();  // every thread has read sh before it is reset
    return b;
}

__device__ __forceinline__ void cta_clear(SelShared &sh) {
    for (int i = threadIdx.x; i < kHistBins; i += kTpThreads) sh.hist[i] = 0ull;
    if (threadIdx.x == 0) {
        sh.cross = INT_MAX;
        sh.lastnz = -1;
    }
    __syncthreads();
}

constexpr int kMaxPieces = 64;   // pieces of one row the summary gather handles
constexpr int kSumBuf = 6144;    // summary entries of one row staged in shared memory

struct ToppShared {
    SelShared sel;
    float alist[kAList];            // the gathered logits (when they fit)
    int aidx[kAList];               // ... and their indices in the row
    union {
        struct {
            float elems[kElemCap];          // the logits of the crossing bin (pass B)
            float queue[kTpWarps][32 * 8];  // one vector slot of one warp (32 lanes x 8 logits)
            int qidx[kTpWarps][32 * 8];     // ... and their indices in the row
            int nidx[kElemCap];             // indices of the nucleus (list building)
        };
        alignas(16) uint32_t sumbuf[kSumBuf];  // the row's summary while the list is gathered
    };
    // The row's pieces: [lo, hi), first vector a0, vectors nv, summary offset.
    int pc_lo[kMaxPieces], pc_hi[kMaxPieces], pc_a0[kMaxPieces], pc_nv[kMaxPieces];
    int pc_off[kMaxPieces + 1];
    float pm[kTpWarps], ps[kTpWarps];  // per-warp statistics (fused)
    uint32_t pf[kTpWarps];
    uint32_t cmax;                  // running max of the row so far (ordered key; fused)
    int n_pc, n_groups;
    int sum_staged;                 // the summary is in sumbuf (else read from global)
    unsigned int cnt8[kTpWarps];
    float m, Z;
    uint32_t flags;
    int n_alist, n_elems, n_nuc;
    unsigned int kmin, kmax;
    unsigned long long zacc;        // fixed-point mass of the top-k set
};
static_assert(sizeof(ToppShared) <= kToppSmem, "top-p shared memory");
static_assert(offsetof(ToppShared, sumbuf) % 16 == 0, "the staged summary is written as 16-byte vectors");

// Every logit >= vmin of a row from global memory, calling `f(l, x)` on
// each (x: its index in the row).
// Warp w streams the w-th eighth of the row's 16-byte vectors (kBatch per
// lane in flight, the next batch loaded while this one is reduced).  For
// every vector slot of a batch the warp first packs its logits >= vmin into
// its shared queue, all lanes converged, then calls f on the queue densely:
// those logits are sparse, and calling f where they lie would run f's path
// once per element slot for nearly every slot.
template <typename T, typename F>
__device__ __forceinline__ void for_row(ToppShared &sh, const T *rowp, int V, float vmin, F &&f) {
    constexpr int P = Elem<T>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *q_w = sh.queue[warp];
    int *qi_w = sh.qidx[warp];
    const Span<T> sp(rowp, 0, V);
    if (tid < sp.a0 - sp.e0) {
        const float l = to_f32(rowp[sp.e0 + tid]);
        if (l >= vmin) f(l, sp.e0 + tid);
    }
    if (tid < sp.e1 - sp.a1) {
        const float l = to_f32(rowp[sp.a1 + tid]);
        if (l >= vmin) f(l, sp.a1 + tid);
    }
    const int per = (sp.nvec + kTpWarps - 1) / kTpWarps;
    const int v0w = min(sp.nvec, warp * per), n = min(sp.nvec, v0w + per) - v0w;
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0) + v0w;
    const uint4 neg = neg_inf_vec<T>();
    constexpr int kStride = 32 * kBatch;
    uint4 q[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) q[u] = lane + u * 32 < n ? ld_stream(vp + lane + u * 32) : neg;
    for (int b0 = 0; b0 < n; b0 += kStride) {  // warp-uniform trip count
        uint4 nq[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = b0 + kStride + u * 32 + lane;
            nq[u] = v < n ? ld_stream(vp + v) : neg;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float h[P];
            unpack<T>(q[u], h);
            uint32_t mask = 0u;
            if (batch_max1<T>(q[u]) >= vmin) {
#pragma unroll
                for (int e = 0; e < P; ++e)
                    if (h[e] >= vmin) mask |= 1u << e;
            }
            const unsigned any = __ballot_sync(0xFFFFFFFFu, mask != 0u);
            if (!any) continue;
            const int cnt = __popc(mask);
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const int tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
            int pos = incl - cnt;
            const int x0 = sp.a0 + (v0w + b0 + u * 32 + lane) * P;
#pragma unroll
            for (int e = 0; e < P; ++e)
                if (mask & (1u << e)) {
                    q_w[pos] = h[e];
                    qi_w[pos] = x0 + e;
                    ++pos;
                }
            __syncwarp();
            for (int i = lane; i < tot; i += 32) f(q_w[i], qi_w[i]);
            __syncwarp();
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) q[u] = nq[u];
    }
}

// Append, for a whole warp, each lane's logits h[e] with bit e of `mask`
// set (indices x0 + e) to the pass-A list: one shared atomic per warp.
template <int N>
__device__ __forceinline__ void alist_append(ToppShared &sh, uint32_t mask, const float (&h)[N],
                                             int x0) {
    const int lane = threadIdx.x & 31;
    if (!__ballot_sync(0xFFFFFFFFu, mask != 0u)) return;
    const int cnt = __popc(mask);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    const int tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    int base = 0;
    if (lane == 31) base = atomicAdd(&sh.n_alist, tot);
    base = __shfl_sync(0xFFFFFFFFu, base, 31);
    int pos = base + incl - cnt;
#pragma unroll
    for (int e = 0; e < N; ++e)
        if (mask & (1u << e)) {
            if (pos < kAList) {
                sh.alist[pos] = h[e];
                sh.aidx[pos] = x0 + e;
            }
            ++pos;
        }
}

// Element e of a raw 16-byte vector as a float (no dynamic register
// indexing: the word is picked by selects).
template <typename T>
__device__ __forceinline__ float elem_of(const uint4 &v, int e) {
    if (Elem<T>::kPerVec == 4) {
        const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
        return __uint_as_float(w);
    }
    const int wi = e >> 1;
    const uint32_t w = wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// alist_append for one batch of kBatch raw vectors per lane: bit u P + e of
// `mask` is element e of vector u, at index x0 + u 32 P + e.  Each lane
// walks only its set bits (typically none or one), so the cost follows the
// candidates, not the batch size.
template <typename T>
__device__ __forceinline__ void alist_append_batch(ToppShared &sh, uint32_t mask,
                                                   const uint4 (&q)[kBatch], int x0) {
    static_assert(kBatch == 4, "vector selects below assume four vectors per lane");
    constexpr int P = Elem<T>::kPerVec;
    if (!mask) return;
    // The list's order does not matter (every later use is a set or an
    // integer sum): each lane reserves its own slots.
    int pos = atomicAdd(&sh.n_alist, __popc(mask));
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1u;
        const int u = i / P, e = i - u * P;
        const uint4 v = u == 0 ? q[0] : u == 1 ? q[1] : u == 2 ? q[2] : q[3];
        if (pos < kAList) {
            sh.alist[pos] = elem_of<T>(v, e);
            sh.aidx[pos] = x0 + u * 32 * P + e;
        }
        ++pos;
    }
}

// The float whose okey<float> is k.
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Statistics of the piece [lo, hi) of the row into this lane's (m_run,
// s_run), as warp_piece_ms computes them, and meanwhile every logit >= (the
// CTA's running max) - tryT appended to the pass-A list: the running max
// never exceeds the row's max m, so every logit >= m - tryT is appended
// (those the list can hold).
template <typename T>
__device__ __forceinline__ void stats_capture(ToppShared &sh, const T *rowp, int lo, int hi,
                                              float c, float tryT, float &m_run, float &s_run,
                                              uint32_t &fl) {
    constexpr int P = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const Span<T> sp(rowp, lo, hi);
    auto scalar = [&](float l) {
        if (l != l) {
            fl |= kFlagNonFinite;
            return;
        }
        if (l > m_run) {
            s_run = __fmul_rn(s_run, ex2(__fmul_rn(__fsub_rn(m_run, l), c)));
            m_run = l;
        }
        if (m_run != kNegInf)
            s_run = __fadd_rn(s_run, ex2(__fmaf_rn(l, c, -__fmul_rn(m_run, c))));
    };
    // Threshold from this lane's and the CTA's running max (either is at
    // most the row's max, so the floor never exceeds m - tryT).  A lane
    // whose max grew publishes it with a shared atomic (rare once the row's
    // top logits have been seen).
    auto floor_now = [&](bool grew) {
        if (grew && m_run > kNegInf) atomicMax(&sh.cmax, okey<float>(m_run));
        const uint32_t ck = *reinterpret_cast<volatile uint32_t *>(&sh.cmax);
        const float ref = ck ? fmaxf(m_run, key_float(ck)) : m_run;
        return ref > kNegInf ? __fsub_rn(ref, tryT) : INFINITY;
    };
    // The ragged ends (< one vector each): counted, then appended if >= the floor.
    auto edge = [&](int n0, int n1) {
        float h[1] = {kNegInf};
        if (lane < n1 - n0) {
            h[0] = to_f32(rowp[n0 + lane]);
            scalar(h[0]);
        }
        const float fl_now = floor_now(true);
        alist_append<1>(sh, (h[0] >= fl_now && h[0] > kNegInf) ? 1u : 0u, h, n0 + lane);
    };
    edge(sp.e0, sp.a0);
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    const uint4 neg = neg_inf_vec<T>();
    constexpr int kStride = 32 * kBatch;
    uint4 q[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) q[u] = lane + u * 32 < sp.nvec ? ld_stream(vp + lane + u * 32) : neg;
    for (int v0 = 0; v0 < sp.nvec; v0 += kStride) {  // warp-uniform trip count
        uint4 nq[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + kStride + u * 32 + lane;
            nq[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        }
        const float bm = batch_max<T>(q);
        const bool nan = bm != bm;
        bool grew = false;
        if (nan) fl |= kFlagNonFinite;
        else if (bm > m_run) {
            s_run = __fmul_rn(s_run, ex2(__fmul_rn(__fsub_rn(m_run, bm), c)));
            m_run = bm;
            grew = true;
        }
        // Floor after this batch's max is counted (so the batch's own top
        // logits are kept); one unpack feeds the sum and the capture mask.
        const float thr = floor_now(grew);
        const bool sum = !nan && m_run != kNegInf;
        const float negmc = -__fmul_rn(m_run, c);
        float2 acc = make_float2(0.0f, 0.0f);
        float h[kBatch * P];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float f[P];
            unpack<T>(q[u], f);
#pragma unroll
            for (int e = 0; e < P; e += 2) {
                const float2 x = fma2(make_float2(f[e], f[e + 1]), make_float2(c, c),
                                      make_float2(negmc, negmc));
                acc = add2(acc, make_float2(ex2(x.x), ex2(x.y)));
            }
#pragma unroll
            for (int e = 0; e < P; ++e) h[u * P + e] = f[e];
        }
        if (sum) s_run = __fadd_rn(s_run, __fadd_rn(acc.x, acc.y));
        // The capture mask only where this lane's batch reaches the floor:
        // past the first batches of a peaked row almost none does.  (A
        // finite floor excludes -inf logits; with no finite max yet the
        // floor is +inf.)
        uint32_t mask = 0u;
        // Once the list has overflowed it is not used: stop filling it.
        if (bm >= thr && *reinterpret_cast<volatile int *>(&sh.n_alist) <= kAList) {
#pragma unroll
            for (int i = 0; i < kBatch * P; ++i)
                if (h[i] >= thr) mask |= 1u << i;
        }
        alist_append_batch<T>(sh, mask, q, sp.a0 + (v0 + lane) * P);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) q[u] = nq[u];
    }
    edge(sp.a1, sp.e1);
}

// One slot of *ctr per lane with `want`, one atomic per warp; the lane's
// slot (meaningless without want).  Every lane of the warp calls it.
__device__ __forceinline__ int warp_reserve(int *ctr, bool want) {
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, want);
    if (!bal) return 0;
    const int lane = threadIdx.x & 31, leader = __ffs(bal) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(ctr, __popc(bal));
    base = __shfl_sync(0xFFFFFFFFu, base, leader);
    return base + __popc(bal & ((1u << lane) - 1u));
}

// Append logit l (index x) to the list where `want` (counted past kAList:
// overflow).  Every lane of the warp calls it.
__device__ __forceinline__ void alist_push(ToppShared &sh, bool want, float l, int x) {
    const int pos = warp_reserve(&sh.n_alist, want);
    if (want && pos < kAList) {
        sh.alist[pos] = l;
        sh.aidx[pos] = x;
    }
}

// Append this lane's logits h[e] with bit e of `mask` set (indices x0 + e):
// one atomic per warp.  Every lane of the warp calls it.
template <int P>
__device__ __forceinline__ void alist_push_mask(ToppShared &sh, uint32_t mask, const float (&h)[P],
                                                int x0) {
    const int lane = threadIdx.x & 31;
    if (!__ballot_sync(0xFFFFFFFFu, mask != 0u)) return;
    const int cnt = __popc(mask);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    int base = 0;
    if (lane == 31) base = atomicAdd(&sh.n_alist, incl);
    int pos = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
#pragma unroll
    for (int e = 0; e < P; ++e)
        if (mask & (1u << e)) {
            if (pos < kAList) {
                sh.alist[pos] = h[e];
                sh.aidx[pos] = x0 + e;
            }
            ++pos;
        }
}

// Row `row`'s pieces into sh.pc_* (the summary's layout).  Returns false
// when the row has more than kMaxPieces pieces.
template <typename T>
__device__ bool stage_pieces(ToppShared &sh, const ToppArgs &a, int row, const T *rowp) {
    const int tid = threadIdx.x, V = a.rows.V;
    const long long rbase = static_cast<long long>(row) * V;
    const long long wf = rbase / a.seg, wl = (rbase + V - 1) / a.seg;
    const int np = static_cast<int>(wl - wf + 1);
    if (np > kMaxPieces) return false;  // uniform
    if (tid < np) {
        int lo, hi;
        piece_bounds(row, V, a.seg, wf + tid, lo, hi);
        const Span<T> sp(rowp, lo, hi);
        sh.pc_lo[tid] = lo;
        sh.pc_hi[tid] = hi;
        sh.pc_a0[tid] = sp.a0;
        sh.pc_nv[tid] = sp.nvec;
    }
    __syncthreads();
    if (tid == 0) {
        int off = 0;
        for (int i = 0; i < np; ++i) {
            sh.pc_off[i] = off;
            off += (sh.pc_nv[i] + kGroupVecs - 1) / kGroupVecs * 32;
        }
        sh.pc_off[np] = off;
        sh.n_pc = np;
    }
    __syncthreads();
    // The summary itself, when it fits (read as 16-byte vectors: piece
    // offsets are multiples of 32 entries and rows start 128-byte aligned).
    const int total = sh.pc_off[np];
    const bool staged = total <= kSumBuf;
    if (staged) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.ws.sum + static_cast<size_t>(row) *
                                                                          a.ws.sum_stride);
        uint4 *dst = reinterpret_cast<uint4 *>(sh.sumbuf);
#pragma unroll 4
        for (int v = tid; v < total / 4; v += kTpThreads) dst[v] = __ldcg(src + v);
    }
    if (tid == 0) sh.sum_staged = staged ? 1 : 0;
    __syncthreads();
    return true;
}

// Calls f(e, entry, valid) for every summary entry of the row (valid) and
// for padding (not valid), every thread the same number of times, so that
// f may use warp collectives; each thread's entries are loaded four at a
// time with several loads in flight.  (Piece offsets are multiples of 32
// entries and rows start 128-byte aligned.)
template <typename F>
__device__ __forceinline__ void for_entries(const ToppShared &sh, const ToppArgs &a, int row,
                                            F &&f) {
    const uint4 *src = sh.sum_staged
                           ? reinterpret_cast<const uint4 *>(sh.sumbuf)
                           : reinterpret_cast<const uint4 *>(a.ws.sum + static_cast<size_t>(row) *
                                                                            a.ws.sum_stride);
    const int nv = sh.pc_off[sh.n_pc] / 4;
    constexpr int kUnroll = 4;
    for (int base = 0; base < nv; base += kUnroll * kTpThreads) {  // uniform
        uint4 w[kUnroll];
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int v = base + r * kTpThreads + threadIdx.x;
            w[r] = v >= nv ? make_uint4(0u, 0u, 0u, 0u) : sh.sum_staged ? src[v] : __ldcg(src + v);
        }
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int v = base + r * kTpThreads + threadIdx.x;
            const bool ok = v < nv;
            f(4 * v, w[r].x, ok);
            f(4 * v + 1, w[r].y, ok);
            f(4 * v + 2, w[r].z, ok);
            f(4 * v + 3, w[r].w, ok);
        }
    }
}

// Every logit >= F of the row into the list: the groups whose summary max
// reaches F are listed first, then read -- the vector holding the max, and
// the group's other vectors only if their bound reaches F -- two groups per
// thread and round, so that each thread's loads are in flight together;
// and the pieces' ragged ends (not summarised).
template <typename T>
__device__ void gather_above(ToppShared &sh, const ToppArgs &a, int row, const T *rowp,
                             float F) {
    constexpr int P = Elem<T>::kPerVec;
    const int tid = threadIdx.x, np = sh.n_pc;
    uint2 *glist = reinterpret_cast<uint2 *>(sh.sel.hist);  // (entry index, entry)
    constexpr int kGList = static_cast<int>(sizeof(sh.sel.hist) / sizeof(uint2));
    if (tid == 0) sh.n_groups = 0;
    __syncthreads();
    for_entries(sh, a, row, [&](int e, uint32_t en, bool ok) {
        const bool want = ok && entry_max(en) >= F;
        const int pos = warp_reserve(&sh.n_groups, want);
        if (want && pos < kGList) glist[pos] = make_uint2(static_cast<uint32_t>(e), en);
    });
    __syncthreads();
    const int ng = sh.n_groups;
    if (ng > kGList) {
        if (tid == 0) sh.n_alist = kAList + 1;  // too many: the row is read instead
        return;
    }
    // Rounds: each thread loads one ragged-end logit (at most P - 1 before
    // a0 and after a1 per piece) and kG groups, then tests them.
    constexpr int kG = 2;
    const int nr = np * 2 * (P - 1);
    const int rounds = max((ng + kG * kTpThreads - 1) / (kG * kTpThreads),
                           (nr + kTpThreads - 1) / kTpThreads);
    for (int k = 0; k < rounds; ++k) {
        float rl = kNegInf;
        int rx = -1;
        const int t = k * kTpThreads + tid;
        if (t < nr) {
            const int i = t / (2 * (P - 1)), r = t - i * 2 * (P - 1);
            const int a0 = sh.pc_a0[i], a1 = a0 + sh.pc_nv[i] * P;
            const int x = r < P - 1 ? sh.pc_lo[i] + r : a1 + (r - (P - 1));
            if (r < P - 1 ? x < a0 : x < sh.pc_hi[i]) {
                rl = to_f32(rowp[x]);
                rx = x;
            }
        }
        uint4 q[kG][kBatch];
        int x0[kG][kBatch];
#pragma unroll
        for (int r = 0; r < kG; ++r) {
            const int g = (k * kG + r) * kTpThreads + tid;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                q[r][u] = neg_inf_vec<T>();
                x0[r][u] = 0;
            }
            if (g >= ng) continue;
            const uint2 ge = glist[g];
            const int e = static_cast<int>(ge.x);
            int i = 0;
            while (i + 1 < np && sh.pc_off[i + 1] <= e) ++i;
            const int j = e - sh.pc_off[i], b = j >> 5, l = j & 31, nv = sh.pc_nv[i];
            const int u1 = entry_vec(ge.y);
            const bool all = entry_rest(ge.y) >= F;
            const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sh.pc_a0[i]);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = b * kGroupVecs + u * 32 + l;
                x0[r][u] = sh.pc_a0[i] + v * P;
                if (v < nv && (all || u == u1)) q[r][u] = __ldcg(vp + v);
            }
        }
        alist_push(sh, rx >= 0 && rl >= F, rl, rx);
#pragma unroll
        for (int r = 0; r < kG; ++r)
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                float h[P];
                unpack<T>(q[r][u], h);
                uint32_t mask = 0u;
#pragma unroll
                for (int e2 = 0; e2 < P; ++e2)
                    if (h[e2] >= F) mask |= 1u << e2;
                alist_push_mask<P>(sh, mask, h, x0[r][u]);
            }
    }
}

// A lower bound of the row's K-th largest logit from its summary: the K-th
// largest group max (one bf16 step below it for fp32 logits, whose maxima
// were rounded up) -- the largest 16-bit key k with at least K group keys
// >= k, by bisection over the keys with block-wide counts.  Returns -inf
// when the summary holds fewer than K finite groups (the ragged ends are
// not summarised).
template <typename T>
__device__ float topk_floor(ToppShared &sh, const ToppArgs &a, int row, int K) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t kneg = sum_key(kNegInf);
    auto count_ge = [&](uint32_t k) {
        unsigned int c = 0u;
        for_entries(sh, a, row, [&](int, uint32_t en, bool ok) { c += ok && (en >> 16) >= k; });
        c = __reduce_add_sync(0xFFFFFFFFu, c);
        if (lane == 0) sh.cnt8[warp] = c;
        __syncthreads();
        unsigned int tot = 0u;
#pragma unroll
        for (int w = 0; w < kTpWarps; ++w) tot += sh.cnt8[w];
        __syncthreads();
        return tot;
    };
    uint32_t lo = kneg + 1u, hi = 0xFFFFu;
    if (count_ge(lo) < static_cast<unsigned int>(K)) return kNegInf;
    while (lo < hi) {  // the largest k in [lo, hi] with count_ge(k) >= K
        const uint32_t mid = (lo + hi + 1u) >> 1;
        if (count_ge(mid) >= static_cast<unsigned int>(K)) lo = mid;
        else hi = mid - 1u;
    }
    uint32_t key = lo;
    if (sizeof(T) == 4) --key;  // one bf16 step below: every such group's max is above it
    return key <= kneg ? kNegInf : sum_value(key);
}

// TOPK: the top-k select is compiled in (its own instantiation, so that the
// top-p-only kernel keeps its registers).  FUSED: the CTA streams its row
// itself (statistics, and the logits near the running max into the list),
// the first kernel of a call; else it takes the rows the warp select
// (select.cu) deferred, with their statistics and summaries from the
// statistics grid (rows.cu), and every other CTA exits.
template <typename T, bool TOPK, bool FUSED>
__global__ void __launch_bounds__(kTpThreads, 3) topp_kernel(const ToppArgs a) {
    // Let the dependent final-draw grid launch once every CTA of this grid
    // has started (it waits for this grid's completion before reading).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(16) unsigned char topp_smem[];
    ToppShared &sh = *reinterpret_cast<ToppShared *>(topp_smem);
    const int row = blockIdx.x, tid = threadIdx.x;
    RowRec *rec = a.ws.rows + row;
    const T *rowp = row_ptr<T>(a.rows, row);
    const float tryT = kToppTry * a.temperature;
    const bool topk = TOPK && a.top_k > 0 && a.top_k < a.rows.V;
    // The list: every logit >= gfloor -- m - tryT (a nucleus usually ends
    // above it), or with top-k (not fused) a lower bound of the K-th largest
    // logit (everything top-k keeps, and so everything top-p then sees).
    float gfloor;
    if (FUSED) {
        // Row statistics: warp w reduces the w-th eighth of the row (a
        // split fixed by V alone), combined in warp order.  Meanwhile, when
        // the row's summary fits the staging buffer, each warp writes its
        // piece's summary there (a store per lane and batch) and the
        // near-max groups are gathered after, from L2 (the CTA has just
        // streamed its row); else the logits near the running max are
        // kept as they stream by.
        const int V = a.rows.V, warp = tid >> 5;
        const int per = ((V + kTpWarps - 1) / kTpWarps + 7) / 8 * 8;
        const int lo = min(V, warp * per), hi = min(V, lo + per);
        int off = 0, total = 0;
        for (int w = 0; w < kTpWarps; ++w) {
            const int l2 = min(V, w * per), h2 = min(V, l2 + per);
            const int g = piece_groups<T>(rowp, l2, h2);
            off += w < warp ? g : 0;
            total += g;
        }
        const bool summ = total <= kSumBuf;
        if (tid == 0) {
            sh.n_alist = 0;
            sh.cmax = 0u;
        }
        if (tid < kTpWarps) {
            const int l2 = min(V, tid * per), h2 = min(V, l2 + per);
            const Span<T> sp(rowp, l2, h2);
            sh.pc_lo[tid] = l2;
            sh.pc_hi[tid] = h2;
            sh.pc_a0[tid] = sp.a0;
            sh.pc_nv[tid] = sp.nvec;
        }
        __syncthreads();
        float pm = kNegInf, ps = 0.0f;
        uint32_t pf = 0u;
        if (summ) warp_piece_ms_sum<T, true>(rowp, lo, hi, a.c, sh.sumbuf + off, pm, ps, pf);
        else stats_capture<T>(sh, rowp, lo, hi, a.c, tryT, pm, ps, pf);
        if ((tid & 31) == 0) sh.pc_off[warp] = off;
        if (tid == 0) {
            sh.pc_off[kTpWarps] = total;
            sh.n_pc = kTpWarps;
            sh.sum_staged = 1;
        }
        warp_reduce_ms(pm, ps, pf, a.c);
        if ((tid & 31) == 0) {
            sh.pm[warp] = pm;
            sh.ps[warp] = ps;
            sh.pf[warp] = pf;
        }
        __syncthreads();
        if (tid == 0) {
            float mm = sh.pm[0], ss = sh.ps[0];
            uint32_t ff = sh.pf[0];
            for (int w = 1; w < kTpWarps; ++w) {
                ms_combine(mm, ss, sh.pm[w], sh.ps[w], a.c);
                ff |= sh.pf[w];
            }
            sh.m = mm;
            sh.Z = ss;
            sh.flags = row_flags(mm, ff);
        }
        __syncthreads();
        // The list: every logit >= m - tryT (unless it overflowed).
        gfloor = __fsub_rn(sh.m, tryT);
        if (summ && sh.flags == 0u) {
            gather_above<T>(sh, a, row, rowp, gfloor);
            __syncthreads();
        }
    } else {
        // The warp select's deferrals (and before it the statistics grid's
        // records and summaries): visible once it has completed.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0) {
            sh.flags = __ldcg(&a.ws.defer[row]);
            if (sh.flags) a.ws.defer[row] = 0u;  // this CTA is its only reader
        }
        __syncthreads();
        if (!sh.flags) return;  // taken by the warp select
        __syncthreads();
        if (tid == 0) {
            sh.m = __ldcg(&rec->m);
            sh.Z = __ldcg(&rec->z_full);
            sh.flags = __ldcg(&rec->flags);
            sh.n_alist = 0;
        }
        __syncthreads();
        gfloor = __fsub_rn(sh.m, tryT);
        if (sh.flags == 0u) {
            bool ok = stage_pieces<T>(sh, a, row, rowp);
            if (ok && topk) gfloor = topk_floor<T>(sh, a, row, a.top_k);
            ok = ok && gfloor > kNegInf;
            if (ok) gather_above<T>(sh, a, row, rowp, gfloor);
            else if (tid == 0) sh.n_alist = kAList + 1;  // no usable bound: the row is read instead
            __syncthreads();
        }
    }
    const float m = sh.m;
    const float Z = sh.Z;
    const uint32_t flags = sh.flags;
    uint32_t lam = 0u;
    float zk = Z;
    if (flags == 0u) {
        const int V = a.rows.V;
        const float c = a.c;
        const float negmc = -__fmul_rn(m, c);
        __syncthreads();
        // What the list holds: every logit >= list_lo (unless it overflowed).
        const float tryfloor = m - tryT;
        float list_lo = sh.n_alist <= kAList ? gfloor : INFINITY;
        uint32_t kfloor = 0u;  // keys below it are not kept (top-k; 0: none)
        // The smallest logit value kfloor keeps (-inf: none).
        auto kval = [&]() {
            return kfloor == 0u ? kNegInf : key_float(sizeof(T) == 2 ? kfloor << 16 : kfloor);
        };
        // The list holds every kept logit >= lo.
        auto in_list = [&](float lo) { return fmaxf(lo, kval()) >= list_lo; };
        float span = 0.0f, inv = 0.0f;
        auto vbin = [&](float l) {
            return min(static_cast<int>(__fmul_rn(__fsub_rn(m, l), inv)), kHistBins - 1);
        };
        auto mass = [&](float l) {
            return __float2ull_rn(__fmul_rn(ex2(__fmaf_rn(l, c, negmc)), kFix));
        };
        // One threshold select over the logits l >= lo with key >= kfloor,
        // each weighing 1 (count) or its fixed-point mass: the largest key
        // lam whose weight from the top reaches `target` (all ties of lam
        // kept).  Pass A histograms the weight by value, uniformly over
        // [lo, m], trying each lo of `los` in turn until the weight above it
        // reaches target (the last one is final); from the list when it
        // holds every logit >= lo, else from the row (refilling the list).
        // Pass B gathers the crossing bin's logits and narrows by key to one.
        // Sets sel_above / sel_hb (weight above lam / at lam, once narrowed
        // to one key: sel_single) and sel_lo (the lo used).
        unsigned long long sel_above = 0ull, sel_hb = 0ull;
        float sel_lo = tryfloor;
        bool sel_single = false;
        auto select = [&](bool count, unsigned long long target, const float *los,
                          int nlo) -> uint32_t {
            auto wt = [&](float l) -> unsigned long long { return count ? 1ull : mass(l); };
            float lo = los[0];
            unsigned long long above = 0ull, hb = 0ull;
            int b0 = 0;
            for (int attempt = 0; attempt < nlo; ++attempt) {
                lo = los[attempt];
                span = __fsub_rn(m, lo);
                inv = span > 0.0f ? static_cast<float>(kHistBins) / span : 0.0f;
                cta_clear(sh.sel);
                if (in_list(lo)) {
                    const int na0 = sh.n_alist;
                    for (int i = tid; i < na0; i += kTpThreads) {
                        const float l = sh.alist[i];
                        if (l >= lo && okey<T>(l) >= kfloor)
                            atomicAdd(&sh.sel.hist[vbin(l)], wt(l));
                    }
                } else {
                    // From the row (it mostly hits L2), keeping every
                    // logit >= lo in the list.
                    if (tid == 0) sh.n_alist = 0;
                    __syncthreads();
                    for_row<T>(sh, rowp, V, lo, [&](float l, int x) {
                        if (okey<T>(l) >= kfloor) atomicAdd(&sh.sel.hist[vbin(l)], wt(l));
                        const int pos = atomicAdd(&sh.n_alist, 1);
                        if (pos < kAList) {
                            sh.alist[pos] = l;
                            sh.aidx[pos] = x;
                        }
                    });
                    __syncthreads();
                    list_lo = sh.n_alist <= kAList ? lo : INFINITY;
                }
                __syncthreads();
                bool crossed;
                b0 = cta_cross(sh.sel, kHistBins, 0ull, target, &above, &hb, &crossed);
                if (crossed) break;
            }
            // Pass B: the logits of bin b0 and their key range.  No logit
            // below vmin can fall into b0 (the margin exceeds any rounding of
            // vbin).
            const float vlo =
                b0 == kHistBins - 1
                    ? lo
                    : __fsub_rn(m, __fmul_rn(static_cast<float>(b0 + 1), span / kHistBins));
            const float vmin =
                fmaxf(lo, vlo - span * 9.5367431640625e-7f - fabsf(vlo) * 9.5367431640625e-7f);
            if (tid == 0) {
                sh.n_elems = 0;
                sh.kmin = 0xFFFFFFFFu;
                sh.kmax = 0u;
            }
            __syncthreads();
            auto in_b0 = [&](float l) {
                return l >= lo && okey<T>(l) >= kfloor && vbin(l) == b0;
            };
            auto take = [&](float l, int) {
                if (in_b0(l)) {
                    const int pos = atomicAdd(&sh.n_elems, 1);
                    if (pos < kElemCap) sh.elems[pos] = l;
                    atomicMin(&sh.kmin, okey<T>(l));
                    atomicMax(&sh.kmax, okey<T>(l));
                }
            };
            if (in_list(lo)) {
                const int na = sh.n_alist;
                for (int i0 = 0; i0 < na; i0 += kTpThreads) {  // uniform
                    const int i = i0 + tid;
                    const float l = i < na ? sh.alist[i] : kNegInf;
                    const bool in = i < na && in_b0(l);
                    const int pos = warp_reserve(&sh.n_elems, in);
                    if (in && pos < kElemCap) sh.elems[pos] = l;
                    const uint32_t kl = __reduce_min_sync(0xFFFFFFFFu, in ? okey<T>(l) : 0xFFFFFFFFu);
                    const uint32_t kh = __reduce_max_sync(0xFFFFFFFFu, in ? okey<T>(l) : 0u);
                    const bool any = __any_sync(0xFFFFFFFFu, in);
                    if ((tid & 31) == 0 && any) {
                        atomicMin(&sh.kmin, kl);
                        atomicMax(&sh.kmax, kh);
                    }
                }
            } else {
                for_row<T>(sh, rowp, V, vmin, take);
            }
            __syncthreads();
            const int ne = sh.n_elems;
            uint32_t klo = sh.kmin, khi = sh.kmax;
            // Narrow by key inside bin b0.
            for (int pass = 0; pass < 4 && khi > klo; ++pass) {
                const unsigned long long W = static_cast<unsigned long long>(khi - klo) + 1ull;
                const int nb = W < static_cast<unsigned long long>(kHistBins) ? static_cast<int>(W)
                                                                               : kHistBins;
                cta_clear(sh.sel);
                auto add = [&](float l) {
                    const uint32_t key = okey<T>(l);
                    if (key < klo || key > khi) return;
                    const int bin =
                        static_cast<int>((static_cast<unsigned long long>(khi - key) * nb) / W);
                    atomicAdd(&sh.sel.hist[bin], wt(l));
                };
                if (ne <= kElemCap) {
                    for (int i = tid; i < ne; i += kTpThreads) add(sh.elems[i]);
                } else {
                    for_row<T>(sh, rowp, V, vmin, [&](float l, int) {
                        if (in_b0(l)) add(l);
                    });
                }
                __syncthreads();
                bool cr;
                unsigned long long ab;
                const int b = cta_cross(sh.sel, nb, above, target, &ab, &hb, &cr);
                above = ab;
                const unsigned long long lo_off =
                    (static_cast<unsigned long long>(b) * W + nb - 1) / nb;
                const unsigned long long hi_off =
                    (static_cast<unsigned long long>(b + 1) * W + nb - 1) / nb - 1;
                const uint32_t nkhi = khi - static_cast<uint32_t>(lo_off);
                klo = khi - static_cast<uint32_t>(hi_off);
                khi = nkhi;
            }
            sel_above = above;
            sel_hb = hb;
            sel_lo = lo;
            sel_single = khi == klo;
            return khi;
        };
        float zsel = Z;          // mass the top-p target is relative to
        float final_lo = tryfloor;  // every kept logit is >= it
        bool have_lam = false;
        if (topk) {
            // Top-k: the K-th largest key by count.  The list holds every
            // logit >= a lower bound of it: one window.  Else (the list
            // overflowed) over windows of the row, from tryT / 4 below the
            // max, doubling to tryT, then 1.5 times wider each (a window
            // that first holds K logits then holds few more, so they mostly
            // fit the list for the passes after); beyond the widest (4608 T
            // below the max) a logit's weight 2^((l - m) c) is zero in fp32.
            float los[11];
            int nlo = 0;
            if (list_lo != INFINITY) {
                los[nlo++] = list_lo;
            } else {
                los[nlo++] = __fsub_rn(m, __fmul_rn(0.25f, tryT));
                los[nlo++] = __fsub_rn(m, __fmul_rn(0.5f, tryT));
                los[nlo++] = tryfloor;
                float wdt = tryT;
                for (int i = 0; i < 7; ++i) {
                    wdt = __fmul_rn(wdt, 1.5f);
                    los[nlo++] = __fsub_rn(m, wdt);
                }
                los[nlo++] = __fsub_rn(m, __fmul_rn(512.0f, tryT));
            }
            const uint32_t tau = select(true, static_cast<unsigned long long>(a.top_k), los, nlo);
            const float lo_k = sel_lo;
            kfloor = tau;
            // Fixed-point mass of the kept set (keys >= tau, all >= lo_k).
            if (tid == 0) sh.zacc = 0ull;
            __syncthreads();
            if (in_list(lo_k)) {
                const int na = sh.n_alist;
                for (int i = tid; i < na; i += kTpThreads) {
                    const float l = sh.alist[i];
                    if (okey<T>(l) >= tau) atomicAdd(&sh.zacc, mass(l));
                }
            } else {
                for_row<T>(sh, rowp, V, lo_k, [&](float l, int) {
                    if (okey<T>(l) >= tau) atomicAdd(&sh.zacc, mass(l));
                });
            }
            __syncthreads();
            zsel = __fmul_rn(__ull2float_rn(sh.zacc), 1.0f / kFix);
            final_lo = lo_k;
            if (!(a.top_p < 1.0f)) {
                lam = tau;
                zk = zsel;
                have_lam = true;
            }
        }
        if (!have_lam) {
            // Top-p over the kept set: the target is top_p of its mass.
            // Logits below c0 = m + T (ln((1 - top_p) zsel / V) - ln 2)
            // cannot be in the nucleus: all of them carry < (1 - top_p) zsel
            // / 2.  Pass A first tries max(c0, m - tryT) (a nucleus usually
            // ends far above c0), then c0.
            const unsigned long long tgt =
                __float2ull_rn(__fmul_rn(__fmul_rn(a.top_p, zsel), kFix));
            const float c0 =
                m + a.temperature *
                        (logf((1.0f - a.top_p) * zsel / static_cast<float>(V)) - 0.69314718f);
            const float cut = fminf(c0, m);
            const float los[2] = {fmaxf(cut, tryfloor), cut};
            lam = select(false, tgt, los, los[0] == cut ? 1 : 2);
            zk = __fmul_rn(__ull2float_rn(sel_single ? sel_above + sel_hb : tgt), 1.0f / kFix);
            final_lo = sel_lo;
        }
        // The nucleus list of a target row for the final draw: the kept
        // logits (keys >= lam, all of them >= lo, so all in pass A's list
        // when it did not overflow), ranked by index, each with the draft
        // logit at the same index (row r's residual pairs target row r
        // with draft row r; the bonus row has no draft row).
        const int R = a.rows.R, kk = a.rows.k;
        const int bq = row / R, rq = row - bq * R;
        if (a.seq.list_draw && rq <= kk) {
            if (tid == 0) sh.n_nuc = 0;
            __syncthreads();
            const int na2 = sh.n_alist;
            // The list holds every kept logit (all are >= final_lo).
            const bool covers = na2 <= kAList && in_list(final_lo);
            if (covers) {
                for (int i0 = 0; i0 < na2; i0 += kTpThreads) {  // uniform
                    const int i = i0 + tid;
                    const bool keep = i < na2 && okey<T>(sh.alist[i]) >= lam;
                    const int pos = warp_reserve(&sh.n_nuc, keep);
                    if (keep && pos < kElemCap) {
                        sh.elems[pos] = sh.alist[i];
                        sh.nidx[pos] = sh.aidx[i];
                    }
                }
            }
            __syncthreads();
            const int nn = sh.n_nuc;
            const bool ok = covers && nn <= min(kElemCap, kNucCap);
            const int tr = bq * (kk + 1) + rq;
            uint4 *L = a.ws.nuc + static_cast<size_t>(tr) * kNucCap;
            // The draft value at each index: a logit, or (draft given as
            // probabilities) q itself.
            const size_t doff = (static_cast<size_t>(bq) * kk + rq) * V;
            const T *drow = rq < kk && !a.seq.qprob ? static_cast<const T *>(a.rows.draft) + doff
                                                    : nullptr;
            const float *dprob = rq < kk && a.seq.qprob
                                     ? static_cast<const float *>(a.rows.draft) + doff
                                     : nullptr;
            if (ok) {
                // Rank by index without comparing every pair: bucket the
                // entries by their index (kTpThreads buckets over [0, V)),
                // scan the bucket counts, place each entry in its bucket,
                // then count the smaller indices inside its bucket alone.
                // The histogram's memory is free now: counts, bucket
                // starts, then the entries in bucket order.
                static_assert(kElemCap % kTpThreads == 0, "entries per thread");
                constexpr int kPerT = kElemCap / kTpThreads;
                int *cnt = reinterpret_cast<int *>(sh.sel.hist);
                int *start = cnt + kTpThreads;
                int *byb = start + kTpThreads;
                static_assert(sizeof(sh.sel.hist) >= sizeof(int) * (2 * kTpThreads + kElemCap),
                              "rank scratch");
                const int lane = tid & 31, warp = tid >> 5;
                cnt[tid] = 0;
                __syncthreads();
                int bk[kPerT], sl[kPerT];
#pragma unroll
                for (int r = 0; r < kPerT; ++r) {
                    const int i = tid + r * kTpThreads;
                    bk[r] = 0;
                    sl[r] = 0;
                    if (i < nn) {
                        bk[r] = static_cast<int>((static_cast<long long>(sh.nidx[i]) * kTpThreads) / V);
                        sl[r] = atomicAdd(&cnt[bk[r]], 1);
                    }
                }
                __syncthreads();
                const int cb = cnt[tid];
                int incl = cb;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (lane == 31) sh.sel.wsum[warp] = static_cast<unsigned long long>(incl);
                __syncthreads();
                int off = 0;
                for (int w = 0; w < warp; ++w) off += static_cast<int>(sh.sel.wsum[w]);
                start[tid] = off + incl - cb;
                __syncthreads();
#pragma unroll
                for (int r = 0; r < kPerT; ++r) {
                    const int i = tid + r * kTpThreads;
                    if (i < nn) byb[start[bk[r]] + sl[r]] = sh.nidx[i];
                }
                __syncthreads();
#pragma unroll
                for (int r = 0; r < kPerT; ++r) {
                    const int i = tid + r * kTpThreads;
                    if (i >= nn) continue;
                    const int xi = sh.nidx[i], s0 = start[bk[r]], nb = cnt[bk[r]];
                    int rank = s0;
                    for (int t = 0; t < nb; ++t) rank += byb[s0 + t] < xi;
                    const float lq = drow ? to_f32(drow[xi]) : dprob ? dprob[xi] : 0.0f;
                    L[rank] = make_uint4(static_cast<uint32_t>(xi), __float_as_uint(sh.elems[i]),
                                         __float_as_uint(lq), 0u);
                }
            }
            if (tid == 0) a.ws.nuc_n[tr] = ok ? nn : -1;
        }
    } else if (tid == 0 && a.seq.list_draw) {
        const int R = a.rows.R, kk = a.rows.k, bq = row / R, rq = row - bq * R;
        if (rq <= kk) a.ws.nuc_n[bq * (kk + 1) + rq] = -1;
    }
    if (tid == 0) {
        RowRec r;
        r.m = m;
        r.z = zk;
        r.lam_key = lam;
        r.arg = 0;
        r.z_full = Z;
        r.flags = flags;
        r.pad[0] = r.pad[1] = 0;
        *rec = r;
    }
    __threadfence();  // the nucleus list, for whichever warp decides the sequence
    __syncthreads();
    if (tid < 32) row_done<T>(a.rows, a.seq, a.ws, a.c, row);
}

// Opt each instantiation into ToppShared's dynamic shared memory, once per
// device.
template <typename K>
bool topp_smem_ok(K kernel, int slot) {
    constexpr int kMaxDev = 64;
    static int done[kMaxDev][8];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    if (__atomic_load_n(&done[dev][slot], __ATOMIC_RELAXED)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kToppSmem) != cudaSuccess)
        return false;
    __atomic_store_n(&done[dev][slot], 1, __ATOMIC_RELAXED);
    return true;
}

template <typename T, bool TOPK, bool FUSED>
int launch_topp_t(const ToppArgs &a, int rows_total, cudaStream_t st) {
    auto kernel = topp_kernel<T, TOPK, FUSED>;
    if (!topp_smem_ok(kernel, (sizeof(T) == 2 ? 1 : 0) + (TOPK ? 2 : 0) + (FUSED ? 4 : 0)))
        return SPEC_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows_total));
    cfg.blockDim = dim3(kTpThreads);
    cfg.dynamicSmemBytes = FUSED ? kToppSmem : sizeof(ToppShared);
    cfg.stream = st;
    // Not fused: launched behind the warp select, which it waits for.
    // Fused: the first kernel of a call, in plain stream order.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = FUSED ? nullptr : attr;
    cfg.numAttrs = FUSED ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, a) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Top-p alone: the fused kernel, one CTA per row.  With top-k: the
// statistics grid (max, normaliser and summary of every row), the warp
// select, then the CTAs of the rows it deferred.  (Measured on the 128-row
// bf16 workloads: the fused kernel is the faster for top-p, where the
// logits it keeps while streaming are all the select needs; for top-k the
// summary finds the K largest without a second read of dense rows.)
template <typename T>
int launch_topp_two(const ToppArgs &in, int rows_total, cudaStream_t st) {
    ToppArgs a = in;
    a.rows_total = rows_total;
    if (a.top_k <= 0) return launch_topp_t<T, false, true>(a, rows_total, st);
    const int dtype = sizeof(T) == 2 ? SPEC_BF16 : SPEC_F32;
    int rc = launch_stream_summary(a.rows, rows_total, a.c, a.ws, dtype, st, &a.seg);
    if (rc != SPEC_OK) return rc;
    rc = launch_select_warp(a, dtype, st);
    if (rc != SPEC_OK) return rc;
    return launch_topp_t<T, true, false>(a, rows_total, st);
}

}  // namespace

int launch_topp_rows(const ToppArgs &a, int rows_total, int dtype, cudaStream_t st) {
    return dtype == SPEC_F32 ? launch_topp_two<float>(a, rows_total, st)
                             : launch_topp_two<uint16_t>(a, rows_total, st);
}

}  // namespace specv
