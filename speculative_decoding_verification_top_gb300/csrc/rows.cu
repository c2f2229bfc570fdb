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
//                 Kinds: 0 stochastic statistics, 1 first argmax, 2
//                 stochastic statistics and the row summaries (the max of
//                 each lane's batch of vectors, stream.cuh) that the top-k
//                 select reads (select.cu, topp.cu).  With top-p or top-k
//                 the decisions wait for the nucleus: the select kernels
//                 take them.  Kind 3 is kind 0 whose deciding warp also
//                 takes the sequence's final draw (draw.cuh, the same steps
//                 as final.cu's warps), so that no final kernel follows: a
//                 whole call on short rows laid out one row per warp, where
//                 a warp decides at most one sequence and the two launches'
//                 latency chain is the call's time.  (It is a kernel of its
//                 own because the draw's registers would cut kind 0's
//                 residency.)

#include "draw.cuh"
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
        if (KIND == 0 || KIND == 3) {
            warp_piece_ms<T>(rowp, lo, hi, a.c, m, s, fl);
            warp_reduce_ms(m, s, fl, a.c);
        } else if (KIND == 2) {
            uint32_t *sum = a.ws.sum + static_cast<size_t>(row) * a.ws.sum_stride +
                            piece_sum_offset<T>(rowp, row, V, a.seg, w);
            warp_piece_ms_sum<T>(rowp, lo, hi, a.c, sum, m, s, fl);
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
            const int bd = row_done<T>(a.rows, a.seq, a.ws, a.c, row);
            if (KIND == 3 && bd >= 0) {
                __syncwarp();  // the decision record, written by several lanes
                draw_run<T, false>(a.fin, bd, 0, a.fin.NS);
            }
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
                    if (KIND != 1) ms_combine(m, s, m2, __ldcg(&pp[i].s), a.c);
                    else arg_combine(m, arg, m2, __ldcg(&pp[i].arg));
                    fl |= __ldcg(&pp[i].flags);
                }
                if (KIND != 1) warp_reduce_ms(m, s, fl, a.c);
                else warp_reduce_arg(m, arg, fl);
                if (lane == 0) write_row(dst, m, s, arg, fl);
                const int bd = row_done<T>(a.rows, a.seq, a.ws, a.c, row);
                if (KIND == 3 && bd >= 0) {
                    __syncwarp();  // the decision record, written by several lanes
                    draw_run<T, false>(a.fin, bd, 0, a.fin.NS);
                }
            }
        }
        s0 += hi - lo;
    }
}

// ------------------------------------------------- grid sizing (host)

// fin (kind 0 only): a whole call's final-draw arguments; when the layout
// is one row per warp, kind 3 runs instead and *drew is set to 1.
template <typename T, int KIND>
int launch_stream_t(const RowView &rows, const SeqArgs &seq, int rows_total, float c,
                    const Workspace &ws, cudaStream_t st, long long *seg_out = nullptr,
                    const FinalArgs *fin = nullptr, int *drew = nullptr) {
    auto kernel = stream_kernel<T, KIND>;
    const int ctas = resident_ctas(kernel, KIND == 2 ? (sizeof(T) == 2 ? 9 : 8)
                                                     : (sizeof(T) == 2 ? 2 : 0) + KIND);
    if (ctas <= 0) return SPEC_ERR_CUDA;
    StreamArgs a;
    a.rows = rows;
    a.seq = seq;
    a.total = static_cast<long long>(rows_total) * rows.V;
    const long long warps = static_cast<long long>(ctas) * kWarps;
    long long seg = (a.total + warps - 1) / warps;
    seg = (seg + 7) / 8 * 8;
    a.seg = seg < kMinSeg ? kMinSeg : seg;
    // Short rows (V <= kMinSeg) in a call that fits the grid: one row per
    // segment, so that the rows' dependent steps (statistics, record,
    // arrival, the decision) run on parallel warps rather than one after
    // another on a single warp -- the latency of a small call.  (A row is
    // then one piece.)
    if (rows.V <= kMinSeg && static_cast<long long>(rows_total) <= warps) a.seg = rows.V;
    a.c = c;
    a.ws = ws;
    a.fin = FinalArgs{};
    const long long used = (a.total + a.seg - 1) / a.seg;
    const unsigned grid = static_cast<unsigned>((used + kWarps - 1) / kWarps);
    if (seg_out) *seg_out = a.seg;
    if (KIND == 0 && fin && a.seg == rows.V) {
        a.fin = *fin;
        if (drew) *drew = 1;
        stream_kernel<T, 3><<<grid, kThreads, 0, st>>>(a);
    } else {
        kernel<<<grid, kThreads, 0, st>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

int launch_stream_rows(const RowView &rows, const SeqArgs &seq, int rows_total, float c,
                       const Workspace &ws, int kind, int dtype, cudaStream_t st,
                       const FinalArgs *fin, int *drew) {
    if (dtype == SPEC_F32)
        return kind == 0 ? launch_stream_t<float, 0>(rows, seq, rows_total, c, ws, st, nullptr,
                                                     fin, drew)
                         : launch_stream_t<float, 1>(rows, seq, rows_total, c, ws, st);
    return kind == 0 ? launch_stream_t<uint16_t, 0>(rows, seq, rows_total, c, ws, st, nullptr,
                                                    fin, drew)
                     : launch_stream_t<uint16_t, 1>(rows, seq, rows_total, c, ws, st);
}

int launch_stream_summary(const RowView &rows, int rows_total, float c, const Workspace &ws,
                          int dtype, cudaStream_t st, long long *seg) {
    SeqArgs none = {};
    none.work = kSeqNone;  // the decisions wait for the nucleus (topp.cu)
    return dtype == SPEC_F32
               ? launch_stream_t<float, 2>(rows, none, rows_total, c, ws, st, seg)
               : launch_stream_t<uint16_t, 2>(rows, none, rows_total, c, ws, st, seg);
}

}  // namespace specv
