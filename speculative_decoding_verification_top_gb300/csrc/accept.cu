// accept.cu -- per-position acceptance rate of a verification batch.
//
// "3.5 Speculative Decoding" (llm-learning-path), "Proof that the output
// distribution is exactly p": position i accepts (once it is tested) with
// probability beta_i = sum_x min(p_i(x), q_i(x)) = 1 - TV(p_i, q_i);
// "Speculative Decoding: Mathematical Foundations, ..." (llms.blog),
// "Acceptance Rate and Total Variation Distance": TV = (1/2) sum |p - q| =
// 1 - sum min(p, q).
//
// accept_kernel   the B k (target row i, draft row i) pairs laid end to
//                 end, one warp per contiguous segment.  It reads the row
//                 records a preceding verify call left (max, normaliser,
//                 nucleus key), so one pass over both rows suffices.  Per
//                 logit pair one exponential: min(p, q) = 2^min(a, b) with
//                 a = l_p c - m_p c - log2 z_p (and b likewise), since 2^x
//                 is increasing.  A pair split over several warps leaves
//                 partials; the last warp to finish it (arrival count, no
//                 waiting) adds them in piece order.
//                 A persistent grid, equal segments that may span pairs (the
//                 row kernel's layout); used without top-p.
// accept_list_kernel, accept_queue_kernel   with top-p.  A target row whose
//                 nucleus list exists holds every x with p(x) > 0 and the
//                 draft logit there, so its pair's sum runs over that list
//                 alone and no row is read: one warp per pair does it.  The
//                 pairs without a list (a nucleus over 1024 tokens) go to a
//                 queue, and the second kernel streams them in 2048-element
//                 chunks over the whole GPU, so one large nucleus does not
//                 leave the call waiting on a single warp.

#include "common.cuh"

namespace specv {
namespace {

struct RowProc {
    float off;     // -(m c) - log2 z: log2 of the probability is l c + off
    uint32_t lam;  // nucleus key (0: every logit kept)
    bool bad;      // the row has a data error
};

__device__ __forceinline__ RowProc row_proc(const RowRec *r, float c) {
    RowProc rp;
    const float m = __ldcg(&r->m), z = __ldcg(&r->z);
    rp.lam = __ldcg(&r->lam_key);
    rp.bad = (__ldcg(&r->flags) & (kFlagNonFinite | kFlagAllNegInf)) != 0u;
    rp.off = __fsub_rn(-__fmul_rn(m, c), log2f(z));
    return rp;
}

// min(p(x), q(x)) from the two logits at x.
template <typename T, bool MASKED>
__device__ __forceinline__ float overlap(float lp, float lq, float c, const RowProc &P,
                                         const RowProc &Q) {
    const float e = ex2(fminf(__fmaf_rn(lp, c, P.off), __fmaf_rn(lq, c, Q.off)));
    if (!MASKED) return e;
    return okey<T>(lp) >= P.lam && okey<T>(lq) >= Q.lam ? e : 0.0f;
}

// This lane's share of sum_x min(p(x), q(x)) over [lo, hi) of the pair.
template <typename T, bool MASKED>
__device__ float warp_piece_overlap(const T *prow, const T *qrow, int lo, int hi, float c,
                                    const RowProc &P, const RowProc &Q) {
    constexpr int VE = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    float acc = 0.0f;
    const bool same = ((reinterpret_cast<uintptr_t>(prow) ^ reinterpret_cast<uintptr_t>(qrow)) &
                       15u) == 0;
    if (!same) {
        // The two rows sit differently against 16-byte boundaries (V * the
        // element size not a multiple of 16): element loads.
        for (int x = lo + lane; x < hi; x += 32)
            acc = __fadd_rn(acc, overlap<T, MASKED>(to_f32(prow[x]), to_f32(qrow[x]), c, P, Q));
        return acc;
    }
    const Span<T> sp(prow, lo, hi);
    if (lane < sp.a0 - sp.e0) {
        const int x = sp.e0 + lane;
        acc = overlap<T, MASKED>(to_f32(prow[x]), to_f32(qrow[x]), c, P, Q);
    }
    const uint4 *vp = reinterpret_cast<const uint4 *>(prow + sp.a0);
    const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + sp.a0);
    const uint4 neg = neg_inf_vec<T>();
    constexpr int kStride = 32 * kBatch;
    uint4 bp[kBatch], bq[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int v = lane + u * 32;
        bp[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
        bq[u] = v < sp.nvec ? ld_stream(vq + v) : neg;
    }
    for (int v0 = lane; v0 < sp.nvec; v0 += kStride) {
        // Next batch of both rows in flight while this one is reduced.
        uint4 np[kBatch], nq[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + kStride + u * 32;
            np[u] = v < sp.nvec ? ld_stream(vp + v) : neg;
            nq[u] = v < sp.nvec ? ld_stream(vq + v) : neg;
        }
        float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float fp[VE], fq[VE];
            unpack<T>(bp[u], fp);
            unpack<T>(bq[u], fq);
#pragma unroll
            for (int e = 0; e < VE; e += 2)
                s = add2(s, make_float2(overlap<T, MASKED>(fp[e], fq[e], c, P, Q),
                                        overlap<T, MASKED>(fp[e + 1], fq[e + 1], c, P, Q)));
        }
        acc = __fadd_rn(acc, __fadd_rn(s.x, s.y));
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            bp[u] = np[u];
            bq[u] = nq[u];
        }
    }
    if (lane < sp.e1 - sp.a1) {
        const int x = sp.a1 + lane;
        acc = __fadd_rn(acc, overlap<T, MASKED>(to_f32(prow[x]), to_f32(qrow[x]), c, P, Q));
    }
    return acc;
}

// Fixed-order warp sum (xor butterfly): the same association on every run.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// sum over a target row's nucleus list of min(p(x), q(x)); entries hold
// (x, target logit, draft logit at x), every target logit kept.  Lane l
// adds entries l, l + 32, ... in that order (eight loads in flight).
template <typename T>
__device__ float list_overlap(const uint4 *L, int n, float c, const RowProc &P, const RowProc &Q) {
    constexpr int kU = 8;
    float acc = 0.0f;
    for (int i0 = threadIdx.x & 31; i0 < n; i0 += 32 * kU) {
        uint4 e[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            e[u] = i0 + 32 * u < n ? __ldcg(L + i0 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (i0 + 32 * u >= n) break;
            const float lp = __uint_as_float(e[u].y), lq = __uint_as_float(e[u].z);
            const float v = ex2(fminf(__fmaf_rn(lp, c, P.off), __fmaf_rn(lq, c, Q.off)));
            acc = __fadd_rn(acc, okey<T>(lq) >= Q.lam ? v : 0.0f);
        }
    }
    return warp_sum(acc);
}

// Write beta (and 1 - beta) of a pair; NaN for a pair with a data error.
__device__ __forceinline__ void write_pair(const AcceptArgs &a, int pair, float sum, bool bad) {
    const float beta = bad ? __int_as_float(0x7FC00000) : fminf(sum, 1.0f);
    a.beta[pair] = beta;
    if (a.tv) a.tv[pair] = __fsub_rn(1.0f, beta);
}

// Record this warp's piece `slot` of a pair split into `pieces`; the warp
// that brings the last piece adds them all in slot order and writes the
// pair.  Partials and the arrival counter are those of the pair's target
// row (idle outside the row kernel; the counter returns to zero).
__device__ __forceinline__ void piece_done(const AcceptArgs &a, int pair, int prow_id, int slot,
                                           int pieces, float sum) {
    const int lane = threadIdx.x & 31;
    if (pieces == 1) {
        if (lane == 0) write_pair(a, pair, sum, false);
        return;
    }
    int last = 0;
    Partial *pp = a.ws.partial + static_cast<size_t>(prow_id) * a.ws.pmax;
    if (lane == 0) {
        pp[slot].s = sum;
        last = arrive(&a.ws.row_ctr[prow_id], 1u) == static_cast<unsigned>(pieces - 1);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    __syncwarp();
    if (!last) return;
    if (lane == 0) a.ws.row_ctr[prow_id] = 0u;
    float v = 0.0f;
    for (int t = lane; t < pieces; t += 32) v = __fadd_rn(v, __ldcg(&pp[t].s));
    v = warp_sum(v);
    if (lane == 0) write_pair(a, pair, v, false);
}

template <typename T, bool MASKED>
__device__ __forceinline__ float pair_piece(const AcceptArgs &a, int b, int i, int lo, int hi,
                                            const RowProc &P, const RowProc &Q) {
    const int V = a.rows.V, k = a.rows.k;
    const T *prow = static_cast<const T *>(a.rows.target) + (static_cast<size_t>(b) * (k + 1) + i) * V;
    const T *qrow = static_cast<const T *>(a.rows.draft) + (static_cast<size_t>(b) * k + i) * V;
    return warp_sum(warp_piece_overlap<T, MASKED>(prow, qrow, lo, hi, a.c, P, Q));
}

// Without top-p: persistent grid, equal segments over the pairs end to end.
template <typename T>
__global__ void __launch_bounds__(kThreads) accept_kernel(const AcceptArgs a) {
    const long long w = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int V = a.rows.V, k = a.rows.k, R = a.rows.R;
    long long s0 = w * a.seg;
    const long long s1 = s0 + a.seg < a.total ? s0 + a.seg : a.total;
    while (s0 < s1) {
        const int pair = static_cast<int>(s0 / V);
        const long long pbase = static_cast<long long>(pair) * V;
        const int lo = static_cast<int>(s0 - pbase);
        const int hi = static_cast<int>(s1 - pbase < V ? s1 - pbase : V);
        s0 += hi - lo;
        const int b = pair / k, i = pair - b * k;
        const int prow_id = b * R + i;
        const RowProc P = row_proc(a.ws.rows + prow_id, a.c);
        const RowProc Q = row_proc(a.ws.rows + b * R + k + 1 + i, a.c);
        const long long wf = pbase / a.seg, wl = (pbase + V - 1) / a.seg;
        if (P.bad || Q.bad) {
            // No row pass: the first piece's warp writes NaN.
            if (w == wf && (threadIdx.x & 31) == 0) write_pair(a, pair, 0.0f, true);
            continue;
        }
        const float sum = pair_piece<T, false>(a, b, i, lo, hi, P, Q);
        piece_done(a, pair, prow_id, static_cast<int>(w - wf), static_cast<int>(wl - wf + 1), sum);
    }
}

// With top-p, step 1: one warp per pair.  A pair whose target row has a
// nucleus list is summed over it; a pair without one is queued for step 2.
template <typename T>
__global__ void __launch_bounds__(kThreads) accept_list_kernel(const AcceptArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int pair = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (pair >= a.pairs) return;
    const int lane = threadIdx.x & 31;
    const int k = a.rows.k, R = a.rows.R;
    const int b = pair / k, i = pair - b * k;
    const RowProc P = row_proc(a.ws.rows + b * R + i, a.c);
    const RowProc Q = row_proc(a.ws.rows + b * R + k + 1 + i, a.c);
    const int tr = b * (k + 1) + i;
    const int nl = min(__ldcg(&a.ws.nuc_n[tr]), kNucCap);
    if (P.bad || Q.bad) {
        if (lane == 0) write_pair(a, pair, 0.0f, true);
    } else if (nl >= 0) {
        const float sum = list_overlap<T>(a.ws.nuc + static_cast<size_t>(tr) * kNucCap, nl, a.c, P, Q);
        if (lane == 0) write_pair(a, pair, sum, false);
    } else if (lane == 0) {
        a.ws.accq[2 + atomicAdd(&a.ws.accq[0], 1u)] = static_cast<uint32_t>(pair);
    }
}

// With top-p, step 2 (a programmatic dependent of step 1): the queued pairs
// in chunks of kMinSeg elements, grid-stride over a resident grid.  The
// last CTA to finish returns the queue to empty.
template <typename T>
__global__ void __launch_bounds__(kThreads) accept_queue_kernel(const AcceptArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int V = a.rows.V, k = a.rows.k, R = a.rows.R;
    const int nch = (V + kMinSeg - 1) / kMinSeg;
    const long long items = static_cast<long long>(__ldcg(&a.ws.accq[0])) * nch;
    const long long warps = static_cast<long long>(gridDim.x) * kWarps;
    for (long long it = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); it < items;
         it += warps) {
        const int q = static_cast<int>(it / nch), chunk = static_cast<int>(it - static_cast<long long>(q) * nch);
        const int pair = static_cast<int>(__ldcg(&a.ws.accq[2 + q]));
        const int b = pair / k, i = pair - b * k;
        const int prow_id = b * R + i;
        const RowProc P = row_proc(a.ws.rows + prow_id, a.c);
        const RowProc Q = row_proc(a.ws.rows + b * R + k + 1 + i, a.c);
        const int lo = chunk * kMinSeg, hi = min(V, lo + kMinSeg);
        const float sum = pair_piece<T, true>(a, b, i, lo, hi, P, Q);
        piece_done(a, pair, prow_id, chunk, nch, sum);
    }
    __syncthreads();
    if (threadIdx.x == 0 && arrive(&a.ws.accq[1], 1u) == gridDim.x - 1) {
        a.ws.accq[0] = 0u;
        a.ws.accq[1] = 0u;
    }
}

template <typename T>
int launch_accept_t(const AcceptArgs &base, bool masked, cudaStream_t st) {
    AcceptArgs a = base;
    const int V = a.rows.V;
    if (!masked) {
        auto kernel = accept_kernel<T>;
        const int ctas = resident_ctas(kernel, sizeof(T) == 2 ? 13 : 12);
        if (ctas <= 0) return SPEC_ERR_CUDA;
        const long long warps = static_cast<long long>(ctas) * kWarps;
        a.total = a.pairs * V;
        long long seg = (a.total + warps - 1) / warps;
        seg = (seg + 7) / 8 * 8;
        a.seg = seg < kMinSeg ? kMinSeg : seg;
        const long long used = (a.total + a.seg - 1) / a.seg;
        kernel<<<static_cast<unsigned>((used + kWarps - 1) / kWarps), kThreads, 0, st>>>(a);
        return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
    }
    auto qkernel = accept_queue_kernel<T>;
    const int ctas = resident_ctas(qkernel, sizeof(T) == 2 ? 15 : 14);
    if (ctas <= 0) return SPEC_ERR_CUDA;
    accept_list_kernel<T><<<static_cast<unsigned>((a.pairs + kWarps - 1) / kWarps), kThreads, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qkernel, a) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

int launch_accept(const AcceptArgs &a, int dtype, bool masked, cudaStream_t st) {
    return dtype == SPEC_F32 ? launch_accept_t<float>(a, masked, st)
                             : launch_accept_t<uint16_t>(a, masked, st);
}

}  // namespace specv
