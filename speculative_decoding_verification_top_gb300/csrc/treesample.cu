// treesample.cu -- stochastic verification of a candidate tree.
//
// "3.5 Speculative Decoding" (llm-learning-path), "Tree verification":
// SpecInfer verifies a sampled tree with a lossless multi-candidate rule
// (named there, not stated).  Reading: a node's children are candidates
// drawn independently from that node's draft row q; at the current node
// they are tried in flattened order, child c accepted iff
//   u_c q(x_c) < p'(x_c),
// p' starting as the node's target row p and becoming, after each rejected
// child, the normalised residual max(0, p' - q) (kept as it is if that
// residual is zero everywhere).  An accepted child becomes the current node;
// when every child is rejected (or there is none) the final token is drawn
// from p' by inverse CDF in token order with the sequence's final uniform.
//
// Row statistics (max, normaliser, nucleus key) of the 2N rows of every
// sequence come from the row kernels.  tree_sample_kernel then walks each
// sequence with one cluster of 8 CTAs (8 SMs), each streaming one slice of
// the vocabulary: a rejected child costs one pass over the node's two rows
// (the residual's normaliser), the final draw one more (the total) plus a
// rescan of one chunk.  p'(x) is never stored: it is rebuilt from p(x), q(x)
// and the normalisers so far, p'_{j+1}(x) = max(0, p'_j(x) - q(x)) /
// S_{j+1}.  Sums run over contiguous per-thread chunks in a fixed order,
// CTA totals are added in rank order through distributed shared memory,
// and the cluster barrier is the only wait.

#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace specv {
namespace {

constexpr int kTsThreads = 256;
constexpr int kTsCluster = 8;  // CTAs per sequence (one cluster), each a slice of V
constexpr int kTsMaxRej = 64;  // residual rounds kept per node (children tried)

struct TsShared {
    int par[SPEC_MAX_TREE_NODES];
    int tok[SPEC_MAX_TREE_NODES];
    int nkids[SPEC_MAX_TREE_NODES];
    float inv_s[kTsMaxRej];   // 1 / S_j of the residual rounds at the current node
    float part[kTsThreads];   // per-thread chunk sums
    float ctot[2];            // this CTA's total of the current pass (two slots, alternating)
    float total, pre;
    int bad_flags;
    int cross, token;
};

// f(lp, lq, y) over y in [x0, x1) in order, on the logits of the two rows at
// y: four 16-byte vectors of each row in flight per step when `vec` (x0 a
// multiple of 4 VE, both rows 16-byte aligned), then the ragged tail.
template <typename T, typename F>
__device__ __forceinline__ void chunk_for(const T *prow, const T *qrow, int x0, int x1, bool vec,
                                          F &&f) {
    constexpr int VE = Elem<T>::kPerVec;
    int y = x0;
    if (vec) {
        for (; y + 4 * VE <= x1; y += 4 * VE) {
            uint4 vp[4], vq[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                vp[u] = __ldg(reinterpret_cast<const uint4 *>(prow + y) + u);
                vq[u] = __ldg(reinterpret_cast<const uint4 *>(qrow + y) + u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float fp[VE], fq[VE];
                unpack<T>(vp[u], fp);
                unpack<T>(vq[u], fq);
#pragma unroll
                for (int e = 0; e < VE; ++e) f(fp[e], fq[e], y + u * VE + e);
            }
        }
    }
    for (; y < x1; ++y) f(to_f32(prow[y]), to_f32(qrow[y]), y);
}

// The processing parameters of one row from its record.
struct RowP {
    float neg, inv;
    uint32_t lam;
};

__device__ __forceinline__ RowP row_p(const RowRec *r, float c) {
    RowP p;
    p.neg = -__fmul_rn(__ldcg(&r->m), c);
    p.inv = __frcp_rn(__ldcg(&r->z));
    p.lam = __ldcg(&r->lam_key);
    return p;
}

// p'(x) after `nrej` residual rounds, from the logits of the two rows at x.
template <typename T>
__device__ __forceinline__ float resid_prob(float lp, float lq, float c, const RowP &P,
                                            const RowP &Q, const float *inv_s, int nrej) {
    float v = proc_prob<T>(lp, c, P.neg, P.inv, P.lam);
    if (nrej == 0) return v;
    const float q = proc_prob<T>(lq, c, Q.neg, Q.inv, Q.lam);
    for (int j = 0; j < nrej; ++j) v = __fmul_rn(fmaxf(__fsub_rn(v, q), 0.0f), inv_s[j]);
    return v;
}

// Block-wide sum of the per-thread values in thread order (fixed
// association); every thread gets the total; sh.part keeps the inputs.
__device__ float block_sum_ordered(TsShared &sh, float v) {
    const int tid = threadIdx.x;
    sh.part[tid] = v;
    __syncthreads();
    if (tid == 0) {
        float s = 0.0f;
        for (int t = 0; t < kTsThreads; ++t) s = __fadd_rn(s, sh.part[t]);
        sh.total = s;
    }
    __syncthreads();
    return sh.total;
}

// The cluster's sum of one value per thread: each CTA adds its threads' in
// thread order, then every CTA adds the CTAs' totals in rank order (read
// from their shared memory), so every thread of the cluster gets the same
// total.  `slot` alternates between passes: a CTA writes a slot again only
// two passes later, after a cluster barrier every reader has passed.
__device__ float cluster_sum(TsShared &sh, cg::cluster_group &cl, float v, int slot) {
    const float mine = block_sum_ordered(sh, v);
    if (threadIdx.x == 0) sh.ctot[slot] = mine;
    cl.sync();
    float s = 0.0f;
    for (int r = 0; r < kTsCluster; ++r) s = __fadd_rn(s, *cl.map_shared_rank(&sh.ctot[slot], r));
    return s;
}

// One cluster of kTsCluster CTAs per sequence; CTA r owns the r-th slice of
// the vocabulary, split into contiguous per-thread chunks.  Every CTA takes
// the same decisions (the same inputs and totals); rank 0 writes the path,
// the CTA whose slice holds the final draw's crossing writes that token.
template <typename T>
__global__ void __launch_bounds__(kTsThreads) tree_sample_kernel(const TreeSampleArgs a) {
    __shared__ TsShared sh;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int b = blockIdx.x / kTsCluster, tid = threadIdx.x, N = a.N, V = a.V, W = a.D + 1;
    const float c = a.c;
    const RowRec *rr = a.ws.rows + static_cast<size_t>(b) * 2 * N;
    const T *tgt = static_cast<const T *>(a.target) + static_cast<size_t>(b) * N * V;
    const T *drf = static_cast<const T *>(a.draft) + static_cast<size_t>(b) * N * V;
    const float *ub = a.uniforms + static_cast<size_t>(b) * N;
    if (tid == 0) sh.bad_flags = 0;
    for (int n = tid; n < N; n += kTsThreads) sh.nkids[n] = 0;
    __syncthreads();
    uint32_t bad = 0;
    for (int n = tid; n < N; n += kTsThreads) {
        const int p = a.parents[n];
        sh.par[n] = p;
        // More children than residual rounds kept: refused as a shape error.
        if (n > 0 && p >= 0 && p < n && atomicAdd(&sh.nkids[p], 1) >= kTsMaxRej)
            bad |= SPEC_DATA_TREE_SHAPE;
        if (n == 0 ? p != -1 : (p < 0 || p >= n)) bad |= SPEC_DATA_TREE_SHAPE;
        const int t = a.node_tokens[static_cast<size_t>(b) * N + n];
        if (n > 0 && (t < 0 || t >= V)) bad |= SPEC_DATA_TOKEN_RANGE;
        sh.tok[n] = t;
        const float u = ub[n];
        if (!(u >= 0.0f && u < 1.0f)) bad |= SPEC_DATA_UNIFORM_RANGE;
        bad |= __ldcg(&rr[n].flags) | __ldcg(&rr[N + n].flags);
    }
    if (bad) atomicOr(&sh.bad_flags, static_cast<int>(bad));
    __syncthreads();
    if (!sh.bad_flags) {
        // Depth bound: a node deeper than D (parents[n] < n: walks end).
        for (int n = tid; n < N; n += kTsThreads) {
            int dep = 0;
            for (int x = n; x != 0; x = sh.par[x]) ++dep;
            if (dep > a.D) atomicOr(&sh.bad_flags, SPEC_DATA_TREE_SHAPE);
        }
        __syncthreads();
    }
    int32_t *ot = a.out_tokens + static_cast<size_t>(b) * W;
    int32_t *op = a.out_path ? a.out_path + static_cast<size_t>(b) * W : nullptr;
    if (sh.bad_flags) {
        // Every CTA of the cluster found the same flags: all leave here.
        if (rank == 0) {
            for (int i = tid; i < W; i += kTsThreads) {
                ot[i] = -1;
                if (op) op[i] = -1;
            }
            if (tid == 0) {
                a.out_num[b] = -1;
                atomicOr(a.ws.err, static_cast<uint32_t>(sh.bad_flags));
            }
        }
        return;
    }
    // This CTA's slice and this thread's chunk of it (multiples of four
    // vectors, so that every chunk starts 16-byte aligned when rows do).
    constexpr int VE = Elem<T>::kPerVec;
    const int span = ((V + kTsCluster - 1) / kTsCluster + 4 * VE - 1) / (4 * VE) * (4 * VE);
    const int s0 = min(V, rank * span), s1 = min(V, s0 + span);
    const int per = ((span + kTsThreads - 1) / kTsThreads + 4 * VE - 1) / (4 * VE) * (4 * VE);
    const int x0 = min(s1, s0 + tid * per), x1 = min(s1, x0 + per);
    int cur = 0, depth = 0, pass = 0;
    if (rank == 0 && tid == 0 && op) op[0] = 0;
    for (;;) {
        const RowP P = row_p(rr + cur, c), Q = row_p(rr + N + cur, c);
        const T *prow = tgt + static_cast<size_t>(cur) * V;
        const T *qrow = drf + static_cast<size_t>(cur) * V;
        const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) &
                          15u) == 0;
        int nrej = 0, next = -1;
        for (int ch = 1; ch < N && next < 0; ++ch) {
            if (sh.par[ch] != cur) continue;  // uniform: every thread reads the same entry
            const int x = sh.tok[ch];
            const float lp = to_f32(prow[x]), lq = to_f32(qrow[x]);
            const float pv = resid_prob<T>(lp, lq, c, P, Q, sh.inv_s, nrej);
            const float qv = proc_prob<T>(lq, c, Q.neg, Q.inv, Q.lam);
            if (__fmul_rn(ub[ch], qv) < pv) {
                next = ch;
                break;
            }
            // Rejected: the normaliser of the next residual.
            float s = 0.0f;
            chunk_for<T>(prow, qrow, x0, x1, vec, [&](float l1, float l2, int) {
                const float v = resid_prob<T>(l1, l2, c, P, Q, sh.inv_s, nrej);
                const float q = proc_prob<T>(l2, c, Q.neg, Q.inv, Q.lam);
                s = __fadd_rn(s, fmaxf(__fsub_rn(v, q), 0.0f));
            });
            const float S = cluster_sum(sh, cl, s, pass++ & 1);
            if (S > 0.0f && nrej < kTsMaxRej) {
                if (tid == 0) sh.inv_s[nrej] = __frcp_rn(S);
                __syncthreads();
                ++nrej;
            }
        }
        if (next >= 0) {
            if (rank == 0 && tid == 0) {
                ot[depth] = sh.tok[next];
                if (op) op[depth + 1] = next;
            }
            ++depth;
            cur = next;
            continue;
        }
        // Final draw from p': the total over fixed chunks, then the slice
        // and the chunk holding u * S, the chunk rescanned in the same order.
        float s = 0.0f;
        chunk_for<T>(prow, qrow, x0, x1, vec, [&](float l1, float l2, int) {
            s = __fadd_rn(s, resid_prob<T>(l1, l2, c, P, Q, sh.inv_s, nrej));
        });
        const int slot = pass & 1;
        const float S = cluster_sum(sh, cl, s, slot);
        const float target = __fmul_rn(ub[0], S);
        // The slice whose running prefix (in rank order, as S was summed)
        // first passes the target; else the last slice with weight.
        float ptot[kTsCluster];
        for (int r = 0; r < kTsCluster; ++r) ptot[r] = *cl.map_shared_rank(&sh.ctot[slot], r);
        // No CTA leaves while another may still read its shared memory.
        cl.sync();
        float pre = 0.0f, pre_last = 0.0f;
        int rc = -1, rlast = -1;
        for (int r = 0; r < kTsCluster; ++r) {
            const float nx = __fadd_rn(pre, ptot[r]);
            if (ptot[r] > 0.0f) {
                rlast = r;
                pre_last = pre;
                if (rc < 0 && nx > target) {
                    rc = r;
                    break;
                }
            }
            pre = nx;
        }
        if (rc < 0) {
            rc = rlast;
            pre = pre_last;
        }
        if (rank == 0 && tid == 0) {
            for (int i = depth + 1; i < W; ++i) {
                ot[i] = -1;
                if (op) op[i] = -1;
            }
            a.out_num[b] = depth;
            if (rc < 0) ot[depth] = -1;
        }
        if (rank != rc) return;
        if (tid == 0) {
            // The first chunk of this slice whose running prefix passes the
            // target, else the last chunk with weight.
            float run = pre;
            int t = 0, lastnz = -1;
            float run_last = pre;
            for (; t < kTsThreads; ++t) {
                const float nx = __fadd_rn(run, sh.part[t]);
                if (sh.part[t] > 0.0f) {
                    lastnz = t;
                    run_last = run;
                    if (nx > target) break;
                }
                run = nx;
            }
            if (t == kTsThreads) {
                t = lastnz;
                run = run_last;
            }
            sh.pre = run;
            sh.cross = t;
            sh.token = -1;
        }
        __syncthreads();
        const int tc = sh.cross;
        if (tid == tc && tc >= 0) {
            float run = sh.pre;
            int tok = -1, last = -1;
            chunk_for<T>(prow, qrow, x0, x1, vec, [&](float l1, float l2, int y) {
                const float w = resid_prob<T>(l1, l2, c, P, Q, sh.inv_s, nrej);
                if (w > 0.0f) {
                    last = y;
                    run = __fadd_rn(run, w);
                    if (tok < 0 && run > target) tok = y;
                }
            });
            sh.token = tok >= 0 ? tok : last;
        }
        __syncthreads();
        if (tid == 0) ot[depth] = sh.token;
        return;
    }
}

}  // namespace

int launch_tree_sample(const TreeSampleArgs &a, int dtype, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B) * kTsCluster);
    cfg.blockDim = dim3(kTsThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kTsCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = dtype == SPEC_F32 ? cudaLaunchKernelEx(&cfg, tree_sample_kernel<float>, a)
                                            : cudaLaunchKernelEx(&cfg, tree_sample_kernel<uint16_t>, a);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
