// rows.cu -- phase 1 of the verification step: per-row statistics.
//
// "3.5 Speculative Decoding" (llm-learning-path), "Notation": p and q are
// the target and draft distributions after temperature (and top-p); the
// accept test and the draws need, for every row, its max m and normaliser
// Z = sum_x 2^((l(x) - m) log2(e)/T), and for the greedy rules its first
// argmax ("Proof that the output distribution is exactly p", last
// paragraph; "Tree verification").
//
// stream_kernel   persistent grid, one warp per equal contiguous segment of
//                 the concatenated rows: perfect load balance, 16-byte
//                 streaming loads with the next batch in flight while the
//                 current one is reduced, no block barriers.  A segment
//                 that ends inside a row leaves a partial; the last warp to
//                 finish a row (atomic arrival count, no waiting) combines
//                 the row's partials into its row record, and the warp that
//                 finishes a sequence's last row (a second arrival count)
//                 takes that sequence's accept decision -- or, in greedy
//                 mode, emits its tokens.
// topp_kernel     one CTA per (row, 16384-element tile); the last CTA of a
//                 row also selects the top-p threshold from the L2-resident
//                 row.

#include "stream.cuh"

namespace specv {
namespace {

// ------------------------------------------------------- stream kernel

template <typename T, int KIND>
__global__ void __launch_bounds__(kThreads) stream_kernel(const StreamArgs a) {
    // Let the dependent final-draw grid launch now: it waits for this grid's
    // completion (griddepcontrol.wait) before reading anything it wrote.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int V = a.rows.V;
    long long s0 = w * a.seg;
    const long long s1 = s0 + a.seg < a.total ? s0 + a.seg : a.total;
    while (s0 < s1) {
        const int row = static_cast<int>(s0 / V);
        const long long rbase = static_cast<long long>(row) * V;
        const int lo = static_cast<int>(s0 - rbase);
        const int hi = static_cast<int>(s1 - rbase < V ? s1 - rbase : V);
        const T *rowp = row_ptr<T>(a.rows, row);

        float m = kNegInf, s = 0.0f;
        int arg = INT_MAX;
        uint32_t fl = 0;
        if (KIND == 0) {
            warp_piece_ms<T>(rowp, lo, hi, a.c, m, s, fl);
            warp_reduce_ms(m, s, fl, a.c);
        } else {
            warp_piece_arg<T>(rowp, lo, hi, m, arg, fl);
            warp_reduce_arg(m, arg, fl);
        }

        const long long wf = rbase / a.seg, wl = (rbase + V - 1) / a.seg;
        const int pieces = static_cast<int>(wl - wf + 1);
        RowRec *dst = a.ws.rows + row;
        if (pieces == 1) {
            if (lane == 0) write_row(dst, m, s, arg, fl);
            row_done<T>(a.rows, a.seq, a.ws, a.c, row);
        } else {
            int last = 0;
            if (lane == 0) {
                Partial p;
                p.m = m;
                p.s = s;
                p.arg = arg;
                p.flags = fl;
                a.ws.partial[static_cast<size_t>(row) * a.ws.pmax + (w - wf)] = p;
                last = arrive(&a.ws.row_ctr[row], 1u) == static_cast<unsigned>(pieces - 1);
            }
            last = __shfl_sync(0xFFFFFFFFu, last, 0);
            __syncwarp();
            if (last) {
                // Every other piece of this row is visible: combine them.
                if (lane == 0) a.ws.row_ctr[row] = 0u;
                m = kNegInf;
                s = 0.0f;
                arg = INT_MAX;
                fl = 0;
                const Partial *pp = a.ws.partial + static_cast<size_t>(row) * a.ws.pmax;
                for (int i = lane; i < pieces; i += 32) {
                    const float m2 = __ldcg(&pp[i].m);
                    if (KIND == 0) ms_combine(m, s, m2, __ldcg(&pp[i].s), a.c);
                    else arg_combine(m, arg, m2, __ldcg(&pp[i].arg));
                    fl |= __ldcg(&pp[i].flags);
                }
                if (KIND == 0) warp_reduce_ms(m, s, fl, a.c);
                else warp_reduce_arg(m, arg, fl);
                if (lane == 0) write_row(dst, m, s, arg, fl);
                row_done<T>(a.rows, a.seq, a.ws, a.c, row);
            }
        }
        s0 += hi - lo;
    }
}

// ---------------------------------------------- top-p (CTA per row tile)

__device__ void block_reduce_ms(float &m, float &s, uint32_t &fl, float c) {
    __shared__ float sm[kWarps], ss[kWarps];
    __shared__ uint32_t sf[kWarps];
    warp_reduce_ms(m, s, fl, c);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sm[warp] = m;
        ss[warp] = s;
        sf[warp] = fl;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < kWarps; ++i) {
            ms_combine(m, s, sm[i], ss[i], c);
            fl |= sf[i];
        }
    }
    __syncthreads();
}

// Visit every element of [lo, hi) once, thread-strided (any order).
template <typename T, typename F>
__device__ __forceinline__ void for_each_elem(const T *rowp, int lo, int hi, F &&f) {
    constexpr int P = Elem<T>::kPerVec;
    const Span<T> sp(rowp, lo, hi);
    const int tid = threadIdx.x;
    if (tid < sp.a0 - sp.e0) f(to_f32(rowp[sp.e0 + tid]));
    const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + sp.a0);
    for (int v = tid; v < sp.nvec; v += kThreads) {
        float f8[P];
        unpack<T>(__ldg(vp + v), f8);
#pragma unroll
        for (int e = 0; e < P; ++e) f(f8[e]);
    }
    if (tid < sp.e1 - sp.a1) f(to_f32(rowp[sp.a1 + tid]));
}

// CTA tile statistics: thread-strided 16-byte loads, one ex2 per logit.
template <typename T>
__device__ __forceinline__ void tile_ms(const T *rowp, int lo, int hi, float c, float &m_run,
                                        float &s_run, uint32_t &fl) {
    for_each_elem<T>(rowp, lo, hi, [&](float l) {
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
    });
}

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
        for_each_elem<T>(rowp, 0, V, [&](float l) {
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
        for (int i = 0; i < warp; ++i) before += wsum[i];
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

template <typename T>
__global__ void __launch_bounds__(kThreads, 4) topp_kernel(const ToppArgs a) {
    const int item = blockIdx.x;
    const int row = item / a.T;
    const int tile = item - row * a.T;
    const T *rowp = row_ptr<T>(a.rows, row);
    const int lo = tile * a.TL;
    const int hi = min(a.rows.V, lo + a.TL);
    __shared__ int s_last;

    float m = kNegInf, s = 0.0f;
    uint32_t fl = 0;
    tile_ms<T>(rowp, lo, hi, a.c, m, s, fl);
    block_reduce_ms(m, s, fl, a.c);
    if (a.T > 1) {
        if (threadIdx.x == 0) {
            Partial p;
            p.m = m;
            p.s = s;
            p.arg = 0;
            p.flags = fl;
            a.ws.partial[static_cast<size_t>(row) * a.ws.pmax + tile] = p;
            __threadfence();
            s_last = atomicAdd(&a.ws.row_ctr[row], 1u) == static_cast<unsigned>(a.T - 1);
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        if (threadIdx.x == 0) a.ws.row_ctr[row] = 0u;
        m = kNegInf;
        s = 0.0f;
        fl = 0;
        if (threadIdx.x < a.T) {
            const Partial *pp = a.ws.partial + static_cast<size_t>(row) * a.ws.pmax + threadIdx.x;
            m = __ldcg(&pp->m);
            s = __ldcg(&pp->s);
            fl = __ldcg(&pp->flags);
        }
        block_reduce_ms(m, s, fl, a.c);
    }
    __shared__ float s_m, s_z;
    __shared__ uint32_t s_fl;
    if (threadIdx.x == 0) {
        s_m = m;
        s_z = s;
        s_fl = row_flags(m, fl);
    }
    __syncthreads();
    uint32_t lam = 0;
    float zk = s_z;
    if (s_fl == 0 && a.top_p < 1.0f)
        topp_select<T>(rowp, a.rows.V, s_m, s_z, a.c, a.temperature, a.top_p, lam, zk);
    if (threadIdx.x == 0) {
        RowRec r;
        r.m = s_m;
        r.z = zk;
        r.lam_key = lam;
        r.arg = 0;
        r.z_full = s_z;
        r.flags = s_fl;
        r.pad[0] = r.pad[1] = 0;
        a.ws.rows[row] = r;
    }
    if (threadIdx.x < 32) row_done<T>(a.rows, a.seq, a.ws, a.c, row);
}

// ------------------------------------------------- grid sizing (host)

template <typename T, int KIND>
int launch_stream_t(const RowView &rows, const SeqArgs &seq, int rows_total, float c,
                    const Workspace &ws, cudaStream_t st) {
    auto kernel = stream_kernel<T, KIND>;
    const int ctas = resident_ctas(kernel, (sizeof(T) == 2 ? 2 : 0) + KIND);
    if (ctas <= 0) return SPEC_ERR_CUDA;
    StreamArgs a;
    a.rows = rows;
    a.seq = seq;
    a.total = static_cast<long long>(rows_total) * rows.V;
    const long long warps = static_cast<long long>(ctas) * kWarps;
    long long seg = (a.total + warps - 1) / warps;
    seg = (seg + 7) / 8 * 8;
    a.seg = seg < kMinSeg ? kMinSeg : seg;
    a.c = c;
    a.ws = ws;
    const long long used = (a.total + a.seg - 1) / a.seg;
    const unsigned grid = static_cast<unsigned>((used + kWarps - 1) / kWarps);
    kernel<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

int launch_stream_rows(const RowView &rows, const SeqArgs &seq, int rows_total, float c,
                       const Workspace &ws, int kind, int dtype, cudaStream_t st) {
    if (dtype == SPEC_F32)
        return kind == 0 ? launch_stream_t<float, 0>(rows, seq, rows_total, c, ws, st)
                         : launch_stream_t<float, 1>(rows, seq, rows_total, c, ws, st);
    return kind == 0 ? launch_stream_t<uint16_t, 0>(rows, seq, rows_total, c, ws, st)
                     : launch_stream_t<uint16_t, 1>(rows, seq, rows_total, c, ws, st);
}

int launch_topp_rows(const ToppArgs &a, int rows_total, int dtype, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>(rows_total) * a.T;
    if (dtype == SPEC_F32) topp_kernel<float><<<grid, kThreads, 0, st>>>(a);
    else topp_kernel<uint16_t><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
