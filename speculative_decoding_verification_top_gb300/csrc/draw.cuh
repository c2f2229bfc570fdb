// draw.cuh -- internal: the final draw of one sequence (residual or bonus
// row), used by final.cu.  "3.5 Speculative Decoding", "The algorithm (one step)",
// steps 3-4: on rejection draw from max(0, p - q) normalised, else the bonus
// token from p_{k+1}; the draw here is an inverse CDF in token order.
#pragma once

#include "common.cuh"

namespace specv {
namespace {

// The rows and processing parameters of one sequence's final draw.  QP:
// the draft row is fp32 probabilities q (qf), used as given.
template <typename T, bool QP>
struct Draw {
    const T *prow;
    const void *qsrc;  // draft row: logits (T), or QP fp32 probabilities
    __device__ __forceinline__ const T *qrow() const { return static_cast<const T *>(qsrc); }
    __device__ __forceinline__ const float *qf() const { return static_cast<const float *>(qsrc); }
    float pneg, pinv, qneg, qinv;
    uint32_t plam, qlam;
    bool use_p;  // weights p (bonus row, or empty residual) instead of max(0, p - q)
    bool vec;    // both rows 16-byte aligned: vector loads
    bool masked; // a nucleus threshold is set (top-p): test each logit's key
};

// The draw of sequence b, from the parameters its decider stored.
template <typename T, bool QP>
__device__ __forceinline__ Draw<T, QP> make_draw(const FinalArgs &a, int b, const SeqRec *rec) {
    const int k = a.k, V = a.V;
    const int j = __ldcg(&rec->j);
    Draw<T, QP> d;
    d.use_p = __ldcg(&rec->use_p) != 0;
    d.prow = static_cast<const T *>(a.target) + (static_cast<size_t>(b) * (k + 1) + j) * V;
    if (d.use_p)
        d.qsrc = d.prow;
    else if (QP)
        d.qsrc = static_cast<const float *>(a.draft) + (static_cast<size_t>(b) * k + j) * V;
    else
        d.qsrc = static_cast<const T *>(a.draft) + (static_cast<size_t>(b) * k + j) * V;
    d.pneg = __ldcg(&rec->pneg);
    d.pinv = __ldcg(&rec->pinv);
    d.plam = __ldcg(&rec->plam);
    d.qneg = __ldcg(&rec->qneg);
    d.qinv = __ldcg(&rec->qinv);
    d.qlam = __ldcg(&rec->qlam);
    d.vec = (reinterpret_cast<uintptr_t>(d.prow) & 15u) == 0 &&
            (reinterpret_cast<uintptr_t>(d.qsrc) & 15u) == 0;
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

// The draft side of a run of VE elements at x, raw: one 16-byte vector of
// logits, or (QP) VE fp32 probabilities in VE / 4 vectors; elements at or
// beyond V read as -inf logits / zero probabilities.
template <typename T, bool QP>
struct QRaw {
    static constexpr int N = QP ? Elem<T>::kPerVec / 4 : 1;
    uint4 v[N];
};

template <typename T, bool QP>
__device__ __forceinline__ void load_q_raw(const Draw<T, QP> &d, int x, int V, QRaw<T, QP> &r) {
    constexpr int VE = Elem<T>::kPerVec;
    if (!QP) {
        r.v[0] = load_raw<T>(d.qrow(), x, V, d.vec);
    } else if (d.vec && x + VE <= V) {
#pragma unroll
        for (int i = 0; i < QRaw<T, QP>::N; ++i)
            r.v[i] = __ldg(reinterpret_cast<const uint4 *>(d.qf() + x) + i);
    } else {
#pragma unroll
        for (int i = 0; i < QRaw<T, QP>::N; ++i) {
            uint32_t e4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int xi = x + 4 * i + e;
                e4[e] = xi < V ? __float_as_uint(d.qf()[xi]) : 0u;
            }
            r.v[i] = make_uint4(e4[0], e4[1], e4[2], e4[3]);
        }
    }
}

template <typename T, bool QP>
__device__ __forceinline__ void unpack_q(const QRaw<T, QP> &r, float (&f)[Elem<T>::kPerVec]) {
    if (!QP) {
        unpack<T>(r.v[0], f);
    } else {
#pragma unroll
        for (int i = 0; i < QRaw<T, QP>::N; ++i) {
            f[4 * i] = __uint_as_float(r.v[i].x);
            f[4 * i + 1] = __uint_as_float(r.v[i].y);
            f[4 * i + 2] = __uint_as_float(r.v[i].z);
            f[4 * i + 3] = __uint_as_float(r.v[i].w);
        }
    }
}

// Draw weights of the VE elements starting at x from their loaded target
// logits lp and draft values lq (logits, or QP probabilities).
template <typename T, bool QP>
__device__ __forceinline__ void weights_from(const Draw<T, QP> &d, int x, int V, float c,
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
                const float q = QP ? lq[e] : __fmul_rn(ex2(__fmaf_rn(lq[e], c, d.qneg)), d.qinv);
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
            const float q = QP ? lq[e] : proc_prob<T>(lq[e], c, d.qneg, d.qinv, d.qlam);
            wv = fmaxf(__fsub_rn(p, q), 0.0f);
        }
        w[e] = x + e < V ? wv : 0.0f;
    }
}


// Element order inside a 1024-element sub-tile: round u, then lane, then the
// VE elements of the lane's vector -- exactly index order.
template <typename T>
__device__ __forceinline__ int sub_x(int t, int u, int lane) {
    return t * kSubW + (u * 32 + lane) * Elem<T>::kPerVec;
}

// The raw vectors of sub-tile t of both draw rows (this lane's share).
template <typename T, bool QP>
struct SubLoad {
    static constexpr int ROUNDS = kSubW / (32 * Elem<T>::kPerVec);
    uint4 p[ROUNDS];
    QRaw<T, QP> q[ROUNDS];
};

template <typename T, bool QP>
__device__ __forceinline__ void subtile_load(const Draw<T, QP> &d, int t, int V,
                                             SubLoad<T, QP> &L) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < SubLoad<T, QP>::ROUNDS; ++u) {
        L.p[u] = load_raw<T>(d.prow, sub_x<T>(t, u, lane), V, d.vec);
        if (!QP) L.q[u].v[0] = d.use_p ? L.p[u] : load_raw<T>(d.qrow(), sub_x<T>(t, u, lane), V, d.vec);
        else if (!d.use_p) load_q_raw<T, QP>(d, sub_x<T>(t, u, lane), V, L.q[u]);
    }
}

// Total draw weight of sub-tile t from its loaded vectors: rounds folded
// in order.
template <typename T, bool QP>
__device__ __forceinline__ float subtile_reduce(const Draw<T, QP> &d, int t, int V, float c,
                                                const SubLoad<T, QP> &L) {
    constexpr int VE = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    float total = 0.0f;
#pragma unroll
    for (int u = 0; u < SubLoad<T, QP>::ROUNDS; ++u) {
        float lp[VE], lq[VE], w[VE];
        unpack<T>(L.p[u], lp);
        unpack_q<T, QP>(L.q[u], lq);
        weights_from<T, QP>(d, sub_x<T>(t, u, lane), V, c, lp, lq, w);
        float v = 0.0f;
#pragma unroll
        for (int e = 0; e < VE; ++e) v = __fadd_rn(v, w[e]);
        float rt;
        warp_excl_scan(v, rt);
        total = __fadd_rn(total, rt);
    }
    return total;
}

// Total draw weight of sub-tile t (all loads issued before any arithmetic).
template <typename T, bool QP>
__device__ float subtile_total(const Draw<T, QP> &d, int t, int V, float c) {
    SubLoad<T, QP> L;
    subtile_load<T, QP>(d, t, V, L);
    return subtile_reduce<T, QP>(d, t, V, c, L);
}

// The smallest x of sub-tile t with w(x) > 0 and pre + C_t(x) > target,
// where C_t is the in-sub-tile cumulative weight computed with the same
// association as subtile_total; else the last x with w(x) > 0.  All loads
// are issued first.
template <typename T, bool QP>
__device__ int subtile_find(const Draw<T, QP> &d, int t, int V, float c, float pre,
                            float target) {
    constexpr int VE = Elem<T>::kPerVec, ROUNDS = kSubW / (32 * VE);
    const int lane = threadIdx.x & 31;
    uint4 rp[ROUNDS];
    QRaw<T, QP> rq[ROUNDS];
#pragma unroll
    for (int u = 0; u < ROUNDS; ++u) {
        rp[u] = load_raw<T>(d.prow, sub_x<T>(t, u, lane), V, d.vec);
        if (!QP) rq[u].v[0] = d.use_p ? rp[u] : load_raw<T>(d.qrow(), sub_x<T>(t, u, lane), V, d.vec);
        else if (!d.use_p) load_q_raw<T, QP>(d, sub_x<T>(t, u, lane), V, rq[u]);
    }
    float R = 0.0f;
    int lastpos = -1, token = -1;
#pragma unroll
    for (int u = 0; u < ROUNDS; ++u) {
        const int x0 = sub_x<T>(t, u, lane);
        float lp[VE], lq[VE], w[VE];
        unpack<T>(rp[u], lp);
        unpack_q<T, QP>(rq[u], lq);
        weights_from<T, QP>(d, x0, V, c, lp, lq, w);
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
        if (token < 0 && hit) token = __shfl_sync(0xFFFFFFFFu, found, __ffs(hit) - 1);
        R = __fadd_rn(R, rt);
    }
    if (token >= 0) return token;
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

__device__ inline Pick pick_subtile(const float *sums, int NS, float u) {
    constexpr int kRegs = 8;  // sums per lane held in registers
    const int lane = threadIdx.x & 31;
    const int per = (NS + 31) / 32;
    const int s0 = min(NS, lane * per), s1 = min(NS, s0 + per);
    Pick p;
    int first = INT_MAX, lastnz = -1;
    float first_pre = 0.0f, lastnz_pre = 0.0f;
    if (per <= kRegs) {
        // NS <= 256 (V <= 262144): each lane's run of sums in registers, one
        // round trip, statically indexed.
        float v[kRegs];
#pragma unroll
        for (int i = 0; i < kRegs; ++i) v[i] = s0 + i < s1 ? __ldcg(sums + s0 + i) : 0.0f;
        float chunk = 0.0f;
#pragma unroll
        for (int i = 0; i < kRegs; ++i)
            if (s0 + i < s1) chunk = __fadd_rn(chunk, v[i]);
        float unused;
        const float base = warp_excl_scan(chunk, unused);
        float run = base;
#pragma unroll
        for (int i = 0; i < kRegs; ++i)
            if (s0 + i < s1) run = __fadd_rn(run, v[i]);
        p.S = __shfl_sync(0xFFFFFFFFu, run, (NS - 1) / per);
        p.target = __fmul_rn(u, p.S);
        run = base;
#pragma unroll
        for (int i = 0; i < kRegs; ++i) {
            if (s0 + i >= s1) break;
            if (first == INT_MAX && __fadd_rn(run, v[i]) > p.target) {
                first = s0 + i;
                first_pre = run;
            }
            if (v[i] > 0.0f) {
                lastnz = s0 + i;
                lastnz_pre = run;
            }
            run = __fadd_rn(run, v[i]);
        }
    } else {
        float chunk = 0.0f;
        for (int s = s0; s < s1; ++s) chunk = __fadd_rn(chunk, __ldcg(sums + s));
        float unused;
        const float base = warp_excl_scan(chunk, unused);
        float run = base;
        for (int s = s0; s < s1; ++s) run = __fadd_rn(run, __ldcg(sums + s));
        p.S = __shfl_sync(0xFFFFFFFFu, run, (NS - 1) / per);
        p.target = __fmul_rn(u, p.S);
        run = base;
        for (int s = s0; s < s1; ++s) {
            const float x = __ldcg(sums + s);
            if (first == INT_MAX && __fadd_rn(run, x) > p.target) {
                first = s;
                first_pre = run;
            }
            if (x > 0.0f) {
                lastnz = s;
                lastnz_pre = run;
            }
            run = __fadd_rn(run, x);
        }
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
    const unsigned nz = __ballot_sync(0xFFFFFFFFu, lastnz >= 0);
    const int src = nz ? 31 - __clz(nz) : 0;
    p.t = max(__shfl_sync(0xFFFFFFFFu, lastnz, src), 0);
    p.pre = __shfl_sync(0xFFFFFFFFu, lastnz_pre, src);
    return p;
}

// Last arrival for sequence b: choose the sub-tile holding u * S, scan it
// for the token and emit the sequence's outputs (a sequence with a data
// error already has its -1 outputs).  Leaves the sequence's counter at
// zero for the next call.
template <typename T, bool QP>
__device__ void finish_sequence(const FinalArgs &a, int b) {
    const int lane = threadIdx.x & 31, k = a.k, V = a.V;
    SeqRec *rec = a.ws.seqs + b;
    if (lane == 0) a.ws.seq_ctr[b] = 0u;
    if (__ldcg(&rec->bad) || __ldcg(&rec->done)) return;  // outputs already written
    Draw<T, QP> d = make_draw<T, QP>(a, b, rec);
    float *sums = a.ws.sub_sums + static_cast<size_t>(b) * a.NS;
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 1) + k];
    Pick pk = pick_subtile(sums, a.NS, u);
    if (!(pk.S > 0.0f) && !d.use_p) {
        // The residual is zero everywhere: draw from p_{j+1} instead.
        d.use_p = true;
        d.qsrc = d.prow;
        for (int s = 0; s < a.NS; ++s) {
            const float st = subtile_total<T, QP>(d, s, V, a.c);
            if (lane == 0) sums[s] = st;
        }
        __threadfence();
        __syncwarp();
        pk = pick_subtile(sums, a.NS, u);
    }
    const int tok = subtile_find<T, QP>(d, pk.t, V, a.c, pk.pre, pk.target);
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

// Sum sub-tiles [t0, t1) of sequence b's draw into its sub-tile sums and
// report them; the last report finishes the sequence.  A sequence with a
// data error, or already drawn, reports without summing.
template <typename T, bool QP>
__device__ __forceinline__ void draw_run(const FinalArgs &a, int b, int t0, int t1) {
    const int lane = threadIdx.x & 31;
    const SeqRec *rec = a.ws.seqs + b;
    if (!__ldcg(&rec->bad) && !__ldcg(&rec->done)) {
        const Draw<T, QP> d = make_draw<T, QP>(a, b, rec);
        float *sums = a.ws.sub_sums + static_cast<size_t>(b) * a.NS;
        for (int t = t0; t < t1; ++t) {
            const float tot = subtile_total<T, QP>(d, t, a.V, a.c);
            if (lane == 0) sums[t] = tot;
        }
    }
    int last = 0;
    if (lane == 0)
        last = arrive(&a.ws.seq_ctr[b], static_cast<unsigned>(t1 - t0)) + (t1 - t0) ==
               static_cast<unsigned>(a.NS);
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    __syncwarp();
    if (last) finish_sequence<T, QP>(a, b);
}

}  // namespace
}  // namespace specv
