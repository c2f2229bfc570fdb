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

#include "draw.cuh"

namespace specv {
namespace {

// Persistent grid: warp w sums its even share of the sub-tiles in the
// flattened (sequence, sub-tile) order, and reports them once per sequence.
template <typename T, bool QP>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 && !QP ? 3 : 2) final_kernel(const FinalArgs a) {
    // Wait until the row kernel has finished and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long w = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const long long total = static_cast<long long>(a.B) * a.NS;
    // Even split over all a.per warps of the grid: warp w takes
    // [w total / W, (w+1) total / W).
    const long long i0 = w * total / a.per;
    const long long i1 = (w + 1) * total / a.per;
    long long i = i0;
    while (i < i1) {
        const int b = static_cast<int>(i / a.NS);
        const int t0 = static_cast<int>(i - static_cast<long long>(b) * a.NS);
        const int t1 = static_cast<int>(i1 - static_cast<long long>(b) * a.NS < a.NS
                                            ? i1 - static_cast<long long>(b) * a.NS
                                            : a.NS);
        i += t1 - t0;
        draw_run<T, QP>(a, b, t0, t1);
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

template <typename T, bool QP>
int launch_final_t(const FinalArgs &in, cudaStream_t st) {
    FinalArgs a = in;
    const int ctas = resident_ctas(final_kernel<T, QP>, (sizeof(T) == 2 ? 5 : 4) + (QP ? 2 : 0));
    if (ctas <= 0) return SPEC_ERR_CUDA;
    // a.per carries the grid's warp count W: every resident warp takes an
    // even share (at least one sub-tile each).
    const long long total = static_cast<long long>(a.B) * a.NS;
    long long warps = static_cast<long long>(ctas) * kWarps;
    if (warps > total) warps = total;
    const long long grid = (warps + kWarps - 1) / kWarps;
    a.per = grid * kWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, final_kernel<T, QP>, a);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

int launch_final(const FinalArgs &a, int dtype, cudaStream_t st) {
    if (dtype == SPEC_F32)
        return a.qprob ? launch_final_t<float, true>(a, st) : launch_final_t<float, false>(a, st);
    return a.qprob ? launch_final_t<uint16_t, true>(a, st) : launch_final_t<uint16_t, false>(a, st);
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
