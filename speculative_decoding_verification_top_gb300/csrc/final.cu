// final.cu -- phase 2 of the verification step: the final draw and emit
// ("3.5 Speculative Decoding", "The algorithm (one step)", steps 3-4; "246
// Speculative Decoding", 3.3; "Speculative Decoding: Mathematical
// Foundations, ...", "The Modified Rejection Sampling Algorithm").
//
// final_kernel  launched as a programmatic dependent of the row kernel,
//               which has already taken every sequence's accept decision.
//               One warp per (sequence, 1024-element sub-tile): it sums the
//               draw weights -- residual max(0, p - q) of the rejecting row,
//               or p of the bonus row -- over its sub-tile with coalesced
//               16-byte loads issued up front and warp-shuffle scans.  The
//               warp that finishes a sequence last (atomic arrival count, no
//               waiting) picks the sub-tile holding u * S and rescans it for
//               the token.  The rescan repeats the sum pass's arithmetic
//               exactly, so the chosen sub-tile always contains the crossing.
// tree_kernel   one CTA per sequence: parent walk of the candidate tree.

#include "common.cuh"

namespace specv {
namespace {

// The rows and processing parameters of one sequence's final draw.
template <typename T>
struct Draw {
    const T *prow, *qrow;
    float pneg, pinv, qneg, qinv;
    uint32_t plam, qlam;
    bool use_p;  // weights p (bonus row, or empty residual) instead of max(0, p - q)
    bool vec;    // both rows 16-byte aligned: vector loads
    bool masked; // a nucleus threshold is set (top-p): test each logit's key
};

// The draw of sequence b, from the parameters its decider stored.
template <typename T>
__device__ __forceinline__ Draw<T> make_draw(const FinalArgs &a, int b, const SeqRec *rec) {
    const int k = a.k, V = a.V;
    const int j = __ldcg(&rec->j);
    Draw<T> d;
    d.use_p = __ldcg(&rec->use_p) != 0;
    d.prow = static_cast<const T *>(a.target) + (static_cast<size_t>(b) * (k + 1) + j) * V;
    d.qrow = d.use_p ? d.prow
                     : static_cast<const T *>(a.draft) + (static_cast<size_t>(b) * k + j) * V;
    d.pneg = __ldcg(&rec->pneg);
    d.pinv = __ldcg(&rec->pinv);
    d.plam = __ldcg(&rec->plam);
    d.qneg = __ldcg(&rec->qneg);
    d.qinv = __ldcg(&rec->qinv);
    d.qlam = __ldcg(&rec->qlam);
    d.vec = (reinterpret_cast<uintptr_t>(d.prow) & 15u) == 0 &&
            (reinterpret_cast<uintptr_t>(d.qrow) & 15u) == 0;
    d.masked = d.plam != 0u || d.qlam != 0u;
    return d;
}

// The raw 16-byte vector of VE logits of one row starting at element x (x a
// multiple of VE); elements at or beyond V read as -inf.
template <typename T>
__device__ __forceinline__ uint4 load_raw(const T *row, int x, int V, bool vec) {
    constexpr int VE = Elem<T>::kPerVec;
    if (vec && x + VE <= V) return __ldg(reinterpret_cast<const uint4 *>(row + x));
    uint32_t w[4];
    if (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = x + e < V ? __float_as_uint(to_f32(row[x + e])) : Elem<float>::kNegInfWord;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = x + 2 * i < V ? __float_as_uint(to_f32(row[x + 2 * i])) >> 16
                                              : 0xFF80u;
            const uint32_t hi = x + 2 * i + 1 < V
                                    ? __float_as_uint(to_f32(row[x + 2 * i + 1])) >> 16
                                    : 0xFF80u;
            w[i] = lo | (hi << 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Load the VE logits of one row starting at element x as floats.
template <typename T>
__device__ __forceinline__ void load_run(const T *row, int x, int V, bool vec,
                                         float (&f)[Elem<T>::kPerVec]) {
    unpack<T>(load_raw<T>(row, x, V, vec), f);
}

// Draw weights of the VE elements starting at x from their loaded logits.
template <typename T>
__device__ __forceinline__ void weights_from(const Draw<T> &d, int x, int V, float c,
                                             const float (&lp)[Elem<T>::kPerVec],
                                             const float (&lq)[Elem<T>::kPerVec],
                                             float (&w)[Elem<T>::kPerVec]) {
    constexpr int VE = Elem<T>::kPerVec;
    if (!d.masked) {
        // No nucleus: every logit is kept.  Residual max(0, p - q) with the
        // subtraction folded into one fused multiply-add.
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            const float ep = ex2(__fmaf_rn(lp[e], c, d.pneg));
            float wv;
            if (d.use_p) {
                wv = __fmul_rn(ep, d.pinv);
            } else {
                const float q = __fmul_rn(ex2(__fmaf_rn(lq[e], c, d.qneg)), d.qinv);
                wv = fmaxf(__fmaf_rn(ep, d.pinv, -q), 0.0f);
            }
            w[e] = x + e < V ? wv : 0.0f;
        }
        return;
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) {
        const float p = proc_prob<T>(lp[e], c, d.pneg, d.pinv, d.plam);
        float wv = p;
        if (!d.use_p) {
            const float q = proc_prob<T>(lq[e], c, d.qneg, d.qinv, d.qlam);
            wv = fmaxf(__fsub_rn(p, q), 0.0f);
        }
        w[e] = x + e < V ? wv : 0.0f;
    }
}

// Draw weights of the VE elements starting at x.
template <typename T>
__device__ __forceinline__ void weights(const Draw<T> &d, int x, int V, float c,
                                        float (&w)[Elem<T>::kPerVec]) {
    constexpr int VE = Elem<T>::kPerVec;
    float lp[VE], lq[VE];
    load_run<T>(d.prow, x, V, d.vec, lp);
    if (!d.use_p) load_run<T>(d.qrow, x, V, d.vec, lq);
    weights_from<T>(d, x, V, c, lp, lq, w);
}

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

// Element order inside a 1024-element sub-tile: round u, then lane, then the
// VE elements of the lane's vector -- exactly index order.
template <typename T>
__device__ __forceinline__ int sub_x(int t, int u, int lane) {
    return t * kSubW + (u * 32 + lane) * Elem<T>::kPerVec;
}

// Total draw weight of sub-tile t: rounds folded in order.  All of the
// sub-tile's loads are issued (as raw vectors) before any arithmetic.
template <typename T>
__device__ float subtile_total(const Draw<T> &d, int t, int V, float c) {
    constexpr int VE = Elem<T>::kPerVec, ROUNDS = kSubW / (32 * VE);
    const int lane = threadIdx.x & 31;
    uint4 rp[ROUNDS], rq[ROUNDS];
#pragma unroll
    for (int u = 0; u < ROUNDS; ++u) {
        rp[u] = load_raw<T>(d.prow, sub_x<T>(t, u, lane), V, d.vec);
        rq[u] = d.use_p ? rp[u] : load_raw<T>(d.qrow, sub_x<T>(t, u, lane), V, d.vec);
    }
    float total = 0.0f;
#pragma unroll
    for (int u = 0; u < ROUNDS; ++u) {
        float lp[VE], lq[VE], w[VE];
        unpack<T>(rp[u], lp);
        unpack<T>(rq[u], lq);
        weights_from<T>(d, sub_x<T>(t, u, lane), V, c, lp, lq, w);
        float v = 0.0f;
#pragma unroll
        for (int e = 0; e < VE; ++e) v = __fadd_rn(v, w[e]);
        float rt;
        warp_excl_scan(v, rt);
        total = __fadd_rn(total, rt);
    }
    return total;
}

// The smallest x of sub-tile t with w(x) > 0 and pre + C_t(x) > target,
// where C_t is the in-sub-tile cumulative weight computed with the same
// association as subtile_total; else the last x with w(x) > 0.
template <typename T>
__device__ int subtile_find(const Draw<T> &d, int t, int V, float c, float pre, float target) {
    constexpr int VE = Elem<T>::kPerVec, ROUNDS = kSubW / (32 * VE);
    const int lane = threadIdx.x & 31;
    float R = 0.0f;
    int lastpos = -1;
#pragma unroll
    for (int u = 0; u < ROUNDS; ++u) {
        const int x0 = sub_x<T>(t, u, lane);
        float w[VE];
        weights<T>(d, x0, V, c, w);
        float v = 0.0f;
#pragma unroll
        for (int e = 0; e < VE; ++e) v = __fadd_rn(v, w[e]);
        float rt;
        const float excl = warp_excl_scan(v, rt);
        float run = 0.0f;
        int found = -1;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            run = __fadd_rn(run, w[e]);
            if (w[e] > 0.0f) {
                lastpos = max(lastpos, x0 + e);
                if (found < 0 && __fadd_rn(pre, __fadd_rn(R, __fadd_rn(excl, run))) > target)
                    found = x0 + e;
            }
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, found >= 0);
        if (hit) return __shfl_sync(0xFFFFFFFFu, found, __ffs(hit) - 1);
        R = __fadd_rn(R, rt);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xFFFFFFFFu, lastpos, o));
    return lastpos;
}

// Selection over a sequence's NS sub-tile sums: total S (a running sum in
// sub-tile order), target = u S, first sub-tile t with pre_t + sum_t >
// target (else the last non-empty one) and its prefix pre_t.
struct Pick {
    float S, target, pre;
    int t;
};

__device__ Pick pick_subtile(const float *sums, int NS, float u) {
    const int lane = threadIdx.x & 31;
    const int per = (NS + 31) / 32;
    const int s0 = min(NS, lane * per), s1 = min(NS, s0 + per);
    float chunk = 0.0f;
    for (int s = s0; s < s1; ++s) chunk = __fadd_rn(chunk, __ldcg(sums + s));
    float unused;
    const float base = warp_excl_scan(chunk, unused);
    float run = base;
    for (int s = s0; s < s1; ++s) run = __fadd_rn(run, __ldcg(sums + s));
    Pick p;
    p.S = __shfl_sync(0xFFFFFFFFu, run, (NS - 1) / per);
    p.target = __fmul_rn(u, p.S);
    int first = INT_MAX, lastnz = -1;
    float first_pre = 0.0f;
    run = base;
    for (int s = s0; s < s1; ++s) {
        const float v = __ldcg(sums + s);
        if (first == INT_MAX && __fadd_rn(run, v) > p.target) {
            first = s;
            first_pre = run;
        }
        if (v > 0.0f) lastnz = s;
        run = __fadd_rn(run, v);
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, first != INT_MAX);
    if (hit) {
        const int src = __ffs(hit) - 1;
        p.t = __shfl_sync(0xFFFFFFFFu, first, src);
        p.pre = __shfl_sync(0xFFFFFFFFu, first_pre, src);
        return p;
    }
    // No sub-tile crosses (only if rounding put u S at the very end): take
    // the last non-empty one, entered at its own prefix.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastnz = max(lastnz, __shfl_xor_sync(0xFFFFFFFFu, lastnz, o));
    p.t = max(lastnz, 0);
    // prefix of p.t: recompute along its owner's walk
    const int owner = p.t / per;
    float pre = base;
    for (int s = s0; s < s1 && s < p.t; ++s) pre = __fadd_rn(pre, __ldcg(sums + s));
    p.pre = __shfl_sync(0xFFFFFFFFu, pre, owner);
    return p;
}

// Last arrival for sequence b: choose the sub-tile holding u * S, scan it
// for the token and emit the sequence's outputs.
template <typename T>
__device__ void finish_sequence(const FinalArgs &a, int b, Draw<T> d) {
    const int lane = threadIdx.x & 31, k = a.k, V = a.V;
    SeqRec *rec = a.ws.seqs + b;
    float *sums = a.ws.sub_sums + static_cast<size_t>(b) * a.NS;
    if (lane == 0) a.ws.seq_ctr[b] = 0u;
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 1) + k];
    Pick pk = pick_subtile(sums, a.NS, u);
    if (!(pk.S > 0.0f) && !d.use_p) {
        // The residual is zero everywhere: draw from p_{j+1} instead.
        d.use_p = true;
        d.qrow = d.prow;
        for (int s = 0; s < a.NS; ++s) {
            const float st = subtile_total<T>(d, s, V, a.c);
            if (lane == 0) sums[s] = st;
        }
        __threadfence();
        __syncwarp();
        pk = pick_subtile(sums, a.NS, u);
    }
    const int tok = subtile_find<T>(d, pk.t, V, a.c, pk.pre, pk.target);
    const int j = __ldcg(&rec->j);
    int32_t *ot = a.out_tokens + static_cast<size_t>(b) * (k + 1);
    if (lane <= k) {
        int32_t v = -1;
        if (lane < j) v = a.draft_tokens[static_cast<size_t>(b) * k + lane];
        else if (lane == j) v = tok;
        ot[lane] = v;
    }
    if (lane == 0) {
        a.out_num[b] = j;
        rec->S = pk.S;
    }
}

// Persistent grid: warp w sums the sub-tiles [w per, (w+1) per) of the
// flattened (sequence, sub-tile) order, and reports them once per sequence.
template <typename T>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 3 : 2) final_kernel(const FinalArgs a) {
    // Wait until the row kernel has finished and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const long long total = static_cast<long long>(a.B) * a.NS;
    const long long i0 = w * a.per;
    const long long i1 = i0 + a.per < total ? i0 + a.per : total;
    long long i = i0;
    while (i < i1) {
        const int b = static_cast<int>(i / a.NS);
        const int t0 = static_cast<int>(i - static_cast<long long>(b) * a.NS);
        const int t1 = static_cast<int>(i1 - static_cast<long long>(b) * a.NS < a.NS
                                            ? i1 - static_cast<long long>(b) * a.NS
                                            : a.NS);
        i += t1 - t0;
        const SeqRec *rec = a.ws.seqs + b;
        if (__ldcg(&rec->bad)) continue;  // outputs already -1 (row kernel)
        const Draw<T> d = make_draw<T>(a, b, rec);
        float *sums = a.ws.sub_sums + static_cast<size_t>(b) * a.NS;
        for (int t = t0; t < t1; ++t) {
            const float tot = subtile_total<T>(d, t, a.V, a.c);
            if (lane == 0) sums[t] = tot;
        }
        int last = 0;
        if (lane == 0)
            last = arrive(&a.ws.seq_ctr[b], static_cast<unsigned>(t1 - t0)) + (t1 - t0) ==
                   static_cast<unsigned>(a.NS);
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        __syncwarp();
        if (last) finish_sequence<T>(a, b, d);
    }
}

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
    if (!s_bad) {
        int key = 0;  // depth * 2048 + (2047 - n) of the best accepted node
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
    const SeqRec *rec = ws.seqs + b;
    if (t < k) {
        if (P) P[static_cast<size_t>(b) * k + t] = rec->P[t];
        if (Q) Q[static_cast<size_t>(b) * k + t] = rec->Q[t];
    }
    if (Z)
        for (int r = t; r < R; r += blockDim.x)
            Z[static_cast<size_t>(b) * R + r] = ws.rows[static_cast<size_t>(b) * R + r].z;
    if (S && t == 0) S[b] = rec->S;
}

int status() { return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

}  // namespace

int launch_final(const FinalArgs &in, int dtype, cudaStream_t st) {
    FinalArgs a = in;
    const int ctas = dtype == SPEC_F32 ? resident_ctas(final_kernel<float>, 4)
                                       : resident_ctas(final_kernel<uint16_t>, 5);
    if (ctas <= 0) return SPEC_ERR_CUDA;
    const long long total = static_cast<long long>(a.B) * a.NS;
    const long long warps = static_cast<long long>(ctas) * kWarps;
    a.per = (total + warps - 1) / warps;
    const long long used = (total + a.per - 1) / a.per;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((used + kWarps - 1) / kWarps));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = dtype == SPEC_F32 ? cudaLaunchKernelEx(&cfg, final_kernel<float>, a)
                                            : cudaLaunchKernelEx(&cfg, final_kernel<uint16_t>, a);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int launch_tree(const TreeArgs &a, cudaStream_t st) {
    tree_kernel<<<a.B, kTreeThreads, 0, st>>>(a);
    return status();
}

int launch_intermediates(const Workspace &ws, int B, int k, float *P, float *Q, float *Z,
                         float *S, cudaStream_t st) {
    intermediates_kernel<<<B, 64, 0, st>>>(ws, B, k, P, Q, Z, S);
    return status();
}

}  // namespace specv
