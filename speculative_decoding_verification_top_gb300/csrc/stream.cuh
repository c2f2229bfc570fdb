// stream.cuh -- internal: a warp's streaming reduction of one piece of a
// logit row (stochastic statistics or first argmax) and the row record
// write, used by the row kernel (rows.cu).
#pragma once

#include "common.cuh"

namespace specv {
namespace {

// ------------------------------------------------- warp piece reductions

// Stochastic statistics of the piece [lo, hi) of a row, accumulated into
// this lane's running (m_run, s_run): s = sum 2^(l c - m c), one ex2 per
// logit; the running sum is rescaled once per batch when the max grows.
template <typename T>
__device__ __forceinline__ void warp_piece_ms(const T *rowp, int lo, int hi, float c,
                                              float &m_run, float &s_run, uint32_t &fl) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int lane = threadIdx.x & 31;
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
    if (lane < sp.a0 - sp.e0) scalar(to_f32(rowp[sp.e0 + lane]));

    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    const uint4 neg = neg_inf_vec<T>();
    constexpr int kStride = 32 * kBatch;
    uint4 q[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int v = lane + u * 32;
        q[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
    }
    for (int v0 = lane; v0 < sp.nvec; v0 += kStride) {
        // Next batch in flight while this one is reduced.
        uint4 nq[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + kStride + u * 32;
            nq[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        }
        const float bm = batch_max<T>(q);
        if (bm != bm) {
            fl |= kFlagNonFinite;
        } else {
            if (bm > m_run) {
                s_run = __fmul_rn(s_run, ex2(__fmul_rn(__fsub_rn(m_run, bm), c)));
                m_run = bm;
            }
            if (m_run != kNegInf) {
                const float negmc = -__fmul_rn(m_run, c);
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    float f[P];
                    unpack<T>(q[u], f);
#pragma unroll
                    for (int e = 0; e < P; e += 2) {
                        // even logits into acc.x, odd into acc.y
                        const float2 x = fma2(make_float2(f[e], f[e + 1]), make_float2(c, c),
                                              make_float2(negmc, negmc));
                        acc = add2(acc, make_float2(ex2(x.x), ex2(x.y)));
                    }
                }
                s_run = __fadd_rn(s_run, __fadd_rn(acc.x, acc.y));
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) q[u] = nq[u];
    }
    if (lane < sp.e1 - sp.a1) scalar(to_f32(rowp[sp.a1 + lane]));
}

// A store that asks L2 to keep the line (evicted after normal lines): the
// summaries are read again right after the statistics grid, which streams
// far more than L2 holds.
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_keep(uint32_t *p, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol));
}

// warp_piece_ms, and the piece's summary: entry b 32 + lane of `sum` gets
// sum_entry of this lane's kBatch vectors of batch b, a store of 4 bytes
// per lane and batch (SMEM: `sum` is in shared memory).
template <typename T, bool SMEM = false>
__device__ __forceinline__ void warp_piece_ms_sum(const T *rowp, int lo, int hi, float c,
                                                  uint32_t *sum, float &m_run, float &s_run,
                                                  uint32_t &fl) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int lane = threadIdx.x & 31;
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
    if (lane < sp.a0 - sp.e0) scalar(to_f32(rowp[sp.e0 + lane]));
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    const uint4 neg = neg_inf_vec<T>();
    constexpr int kStride = 32 * kBatch;
    uint4 q[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) q[u] = lane + u * 32 < sp.nvec ? ld_stream(vp + lane + u * 32) : neg;
    uint32_t *sl = sum + lane;
    const uint64_t keep = l2_keep_policy();
    for (int v0 = 0; v0 < sp.nvec; v0 += kStride, sl += 32) {
        uint4 nq[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + kStride + u * 32 + lane;
            nq[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        }
        float mu[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) mu[u] = batch_max1<T>(q[u]);
        const float bm = max_nan(max_nan(mu[0], mu[1]), max_nan(mu[2], mu[3]));
        if (SMEM) *sl = sum_entry(mu);
        else st_keep(sl, sum_entry(mu), keep);
        if (bm != bm) {
            fl |= kFlagNonFinite;
        } else {
            if (bm > m_run) {
                s_run = __fmul_rn(s_run, ex2(__fmul_rn(__fsub_rn(m_run, bm), c)));
                m_run = bm;
            }
            if (m_run != kNegInf) {
                const float negmc = -__fmul_rn(m_run, c);
                float2 acc = make_float2(0.0f, 0.0f);
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
                }
                s_run = __fadd_rn(s_run, __fadd_rn(acc.x, acc.y));
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) q[u] = nq[u];
    }
    if (lane < sp.e1 - sp.a1) scalar(to_f32(rowp[sp.a1 + lane]));
}

// Max and first argmax of the piece [lo, hi), into this lane's (best, idx).
template <typename T>
__device__ __forceinline__ void warp_piece_arg(const T *rowp, int lo, int hi, float &best,
                                               int &idx, uint32_t &fl) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int lane = threadIdx.x & 31;
    auto scalar = [&](float l, int i) {
        if (l != l) fl |= kFlagNonFinite;
        else if (l > best) {
            best = l;
            idx = i;
        }
    };
    if (lane < sp.a0 - sp.e0) scalar(to_f32(rowp[sp.e0 + lane]), sp.e0 + lane);

    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    const uint4 neg = neg_inf_vec<T>();
    constexpr int kStride = 32 * kBatch;
    uint4 q[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int v = lane + u * 32;
        q[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
    }
    for (int v0 = lane; v0 < sp.nvec; v0 += kStride) {
        uint4 nq[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + kStride + u * 32;
            nq[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        }
        const float bm = batch_max<T>(q);
        if (bm != bm) {
            fl |= kFlagNonFinite;
        } else if (bm > best) {
            int found = INT_MAX;
#pragma unroll
            for (int u = kBatch - 1; u >= 0; --u) {
                float f[P];
                unpack<T>(q[u], f);
#pragma unroll
                for (int e = P - 1; e >= 0; --e)
                    if (f[e] == bm) found = sp.a0 + (v0 + u * 32) * P + e;
            }
            best = bm;
            idx = found;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) q[u] = nq[u];
    }
    if (lane < sp.e1 - sp.a1) scalar(to_f32(rowp[sp.a1 + lane]), sp.a1 + lane);
}

__device__ __forceinline__ void write_row(RowRec *dst, float m, float s, int arg, uint32_t fl) {
    RowRec r;
    r.m = m;
    r.z = s;
    r.lam_key = 0;
    r.arg = arg;
    r.z_full = s;
    r.flags = row_flags(m, fl);
    r.pad[0] = r.pad[1] = 0;
    *dst = r;
}

}  // namespace
}  // namespace specv
