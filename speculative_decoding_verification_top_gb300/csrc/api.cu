// api.cu -- the C ABI of libspecverify.so (declared in include/spec_verify.h):
// argument validation, workspace layout and kernel dispatch.  No compute.

#include "common.cuh"

#define SPEC_EXPORT extern "C" __attribute__((visibility("default")))

namespace specv {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int subs_for(int V) { return (V + kSubW - 1) / kSubW; }
// Partial slots per row: a row of V elements meets at most ceil(V / seg) + 1
// warp segments (seg >= kMinSeg).
int pmax_for(int V) { return (V + kMinSeg - 1) / kMinSeg + 2; }

// Carve the workspace; returns the bytes needed (base may be null).
// `chain`: a chain call (rows_per_seq = 2k+1), which also needs the top-p
// nucleus lists of its B (k+1) target rows; a tree call does not.
// `capture`: the row summaries and deferral flags of the top-k path, laid
// out last, so that calls without top-k need only what comes before.
size_t carve(void *base, int B, int rows_per_seq, int V, Workspace *ws, bool chain,
             bool capture) {
    const size_t rows = static_cast<size_t>(B) * rows_per_seq;
    const int pmax = pmax_for(V), NS = subs_for(V);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return static_cast<char *>(base) + o;
    };
    char *err = take(kAlign);
    char *row_ctr = take(rows * sizeof(uint32_t));
    char *seq_rows = take(static_cast<size_t>(B) * sizeof(uint32_t));
    char *seq_ctr = take(static_cast<size_t>(B) * sizeof(uint32_t));
    char *partial = take(rows * pmax * sizeof(Partial));
    char *rowrec = take(rows * sizeof(RowRec));
    char *subs = take(static_cast<size_t>(B) * NS * sizeof(float));
    char *seqs = take(static_cast<size_t>(B) * sizeof(SeqRec));
    const size_t trows = chain ? static_cast<size_t>(B) * ((rows_per_seq + 1) / 2) : 0;
    char *nuc_n = take(trows * sizeof(int32_t));
    char *nuc = take(trows * kNucCap * sizeof(uint4));
    const size_t pairs = chain ? static_cast<size_t>(B) * ((rows_per_seq - 1) / 2) : 0;
    char *accq = take(chain ? (pairs + 2) * sizeof(uint32_t) : 0);
    char *sum = take(capture ? rows * sum_stride_for(V) * sizeof(uint32_t) : 0);
    char *defer = take(capture ? rows * sizeof(uint32_t) : 0);
    if (ws) {
        ws->err = reinterpret_cast<uint32_t *>(err);
        ws->row_ctr = reinterpret_cast<uint32_t *>(row_ctr);
        ws->seq_rows = reinterpret_cast<uint32_t *>(seq_rows);
        ws->seq_ctr = reinterpret_cast<uint32_t *>(seq_ctr);
        ws->partial = reinterpret_cast<Partial *>(partial);
        ws->rows = reinterpret_cast<RowRec *>(rowrec);
        ws->sub_sums = reinterpret_cast<float *>(subs);
        ws->seqs = reinterpret_cast<SeqRec *>(seqs);
        ws->nuc_n = reinterpret_cast<int32_t *>(nuc_n);
        ws->nuc = reinterpret_cast<uint4 *>(nuc);
        ws->accq = reinterpret_cast<uint32_t *>(accq);
        ws->sum = reinterpret_cast<uint32_t *>(sum);
        ws->sum_stride = sum_stride_for(V);
        ws->defer = reinterpret_cast<uint32_t *>(defer);
        ws->pmax = pmax;
    }
    return off;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool chain_sizes_ok(int B, int k, int V) {
    if (B < 0 || k < 1 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return false;
    const long long rows = static_cast<long long>(B) * (2 * k + 1);
    return rows * pmax_for(V) < INT_MAX && static_cast<long long>(B) * subs_for(V) * 32 < INT_MAX;
}

bool tree_sizes_ok(int B, int N, int V) {
    if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V) return false;
    return static_cast<long long>(B) * N * pmax_for(V) < INT_MAX;
}

struct ChainPlan {
    RowView rows;
    SeqArgs seq;
    Workspace ws;
    FinalArgs fin;
    int stoch, dtype, rows_total, use_topp, top_k;
    float c, temperature, top_p;
    cudaStream_t st;
    int inline_draw;  // the rows kernel also draws (short rows, a whole call)
};

// qprob: draft_logits holds fp32 probabilities q [B, k, V], used as given
// (stochastic mode only); the rows streamed are the k+1 target rows.
int plan_chain(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
               const float *uniforms, int B, int k, int V, float temperature, float top_p,
               int mode, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
               void *workspace, size_t workspace_bytes, spec_stream_t stream, ChainPlan *plan,
               bool qprob = false, int top_k = 0) {
    if (mode != SPEC_STOCHASTIC && mode != SPEC_GREEDY) return SPEC_ERR_MODE;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;  // nothing is read or written: any pointer will do
    const bool stoch = mode == SPEC_STOCHASTIC;
    if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted || !workspace)
        return SPEC_ERR_NULL;
    if (stoch && (!draft_logits || !uniforms)) return SPEC_ERR_NULL;
    if (stoch && (!(temperature > 0.0f) || !std::isfinite(temperature) || !(top_p > 0.0f) ||
                  !(top_p <= 1.0f)))
        return SPEC_ERR_PARAM;
    const size_t esz = dtype == SPEC_F32 ? 4 : 2;
    if (!aligned(target_logits, esz) || (stoch && !aligned(draft_logits, qprob ? 4 : esz)) ||
        !aligned(draft_tokens, 4) || (stoch && !aligned(uniforms, 4)) ||
        !aligned(out_tokens, 4) || !aligned(out_num_accepted, 4) || !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    const bool topk_on = stoch && top_k > 0 && top_k < V;
    if (workspace_bytes < carve(nullptr, B, 2 * k + 1, V, nullptr, true, topk_on))
        return SPEC_ERR_WORKSPACE;

    plan->stoch = stoch;
    plan->dtype = dtype;
    plan->temperature = stoch ? temperature : 1.0f;
    plan->top_p = stoch ? top_p : 1.0f;
    // top_k <= 0 or >= V keeps every logit (no top-k).
    plan->top_k = stoch && top_k > 0 && top_k < V ? top_k : 0;
    plan->use_topp = stoch && (top_p < 1.0f || plan->top_k > 0);
    plan->c = static_cast<float>(1.4426950408889634 / static_cast<double>(plan->temperature));
    plan->st = reinterpret_cast<cudaStream_t>(stream);
    carve(workspace, B, 2 * k + 1, V, &plan->ws, true, topk_on);

    RowView &rv = plan->rows;
    rv.target = target_logits;
    rv.draft = draft_logits;
    rv.V = V;
    rv.k = k;
    rv.R = stoch && !qprob ? 2 * k + 1 : k + 1;
    rv.draft_rows_from = k + 1;
    rv.tgt_rows_per_seq = k + 1;
    plan->rows_total = B * rv.R;

    FinalArgs &fa = plan->fin;
    fa.target = target_logits;
    fa.draft = draft_logits;
    fa.qprob = qprob ? 1 : 0;
    fa.draft_tokens = draft_tokens;
    fa.uniforms = uniforms;
    fa.B = B;
    fa.k = k;
    fa.V = V;
    fa.NS = subs_for(V);
    fa.c = plan->c;
    fa.out_tokens = out_tokens;
    fa.out_num = out_num_accepted;
    fa.ws = plan->ws;

    SeqArgs &sq = plan->seq;
    sq.work = stoch ? kSeqDecide : kSeqGreedy;
    sq.list_draw = plan->use_topp ? 1 : 0;
    sq.qprob = qprob ? 1 : 0;
    sq.draft_tokens = draft_tokens;
    sq.uniforms = uniforms;
    sq.out_tokens = out_tokens;
    sq.out_num = out_num_accepted;
    plan->inline_draw = 0;
    return SPEC_OK;
}

// Row statistics and accept decisions.  With top-p one kernel does both
// for every row (statistics, then the nucleus), and takes the decisions.
// A whole stochastic call (logits form, no top-p or top-k) may also draw
// there: on short rows laid out one row per warp, the deciding warp takes
// its sequence's final draw and p.inline_draw is set.
int launch_chain_rows(ChainPlan &p, bool whole) {
    const bool offer = whole && p.stoch && !p.use_topp && !p.fin.qprob;
    p.inline_draw = 0;
    if (!p.use_topp)
        return launch_stream_rows(p.rows, p.seq, p.rows_total, p.c, p.ws, p.stoch ? 0 : 1,
                                  p.dtype, p.st, offer ? &p.fin : nullptr, &p.inline_draw);
    ToppArgs ta;
    ta.rows = p.rows;
    ta.seq = p.seq;
    ta.c = p.c;
    ta.temperature = p.temperature;
    ta.top_p = p.top_p;
    ta.top_k = p.top_k;
    ta.ws = p.ws;
    return launch_topp_rows(ta, p.rows_total, p.dtype, p.st);
}

// Greedy verification completes inside the row kernel: nothing to finish.
int launch_chain_finish(const ChainPlan &p) {
    return p.stoch && !p.inline_draw ? launch_final(p.fin, p.dtype, p.st) : SPEC_OK;
}

}  // namespace

size_t chain_workspace_bytes(int B, int k, int V, bool topk) {
    return carve(nullptr, B, 2 * k + 1, V, nullptr, true, topk);
}

}  // namespace specv

using namespace specv;

SPEC_EXPORT int spec_verify_workspace_size(int B, int k, int V, size_t *bytes) {
    if (!bytes) return SPEC_ERR_NULL;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    *bytes = carve(nullptr, B, 2 * k + 1, V, nullptr, true, true);
    return SPEC_OK;
}

SPEC_EXPORT int spec_verify_tree_workspace_size(int B, int N, int V, size_t *bytes) {
    if (!bytes) return SPEC_ERR_NULL;
    if (!tree_sizes_ok(B, N, V)) return SPEC_ERR_SHAPE;
    *bytes = carve(nullptr, B, N, V, nullptr, false, false);
    return SPEC_OK;
}

SPEC_EXPORT int spec_verify_workspace_init(void *workspace, size_t bytes, spec_stream_t stream) {
    if (!workspace) return SPEC_ERR_NULL;
    return cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
}

SPEC_EXPORT int spec_verify_sample(const void *target_logits, const void *draft_logits,
                                   const int32_t *draft_tokens, const float *uniforms, int B,
                                   int k, int V, float temperature, float top_p, int mode,
                                   int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                                   void *workspace, size_t workspace_bytes,
                                   spec_stream_t stream) {
    ChainPlan plan;
    int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V, temperature,
                        top_p, mode, dtype, out_tokens, out_num_accepted, workspace,
                        workspace_bytes, stream, &plan);
    if (rc != SPEC_OK || B == 0) return rc;
    rc = launch_chain_rows(plan, true);
    if (rc != SPEC_OK) return rc;
    return launch_chain_finish(plan);
}

SPEC_EXPORT int spec_verify_sample_topk(const void *target_logits, const void *draft_logits,
                                        const int32_t *draft_tokens, const float *uniforms, int B,
                                        int k, int V, float temperature, float top_p, int top_k,
                                        int mode, int dtype, int32_t *out_tokens,
                                        int32_t *out_num_accepted, void *workspace,
                                        size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V, temperature,
                        top_p, mode, dtype, out_tokens, out_num_accepted, workspace,
                        workspace_bytes, stream, &plan, false, top_k);
    if (rc != SPEC_OK || B == 0) return rc;
    rc = launch_chain_rows(plan, true);
    if (rc != SPEC_OK) return rc;
    return launch_chain_finish(plan);
}

SPEC_EXPORT int spec_verify_sample_rows(const void *target_logits, const void *draft_logits,
                                        const int32_t *draft_tokens, const float *uniforms,
                                        int B, int k, int V, float temperature, float top_p,
                                        int mode, int dtype, int32_t *out_tokens,
                                        int32_t *out_num_accepted, void *workspace,
                                        size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    const int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V,
                              temperature, top_p, mode, dtype, out_tokens, out_num_accepted,
                              workspace, workspace_bytes, stream, &plan);
    if (rc != SPEC_OK || B == 0) return rc;
    return launch_chain_rows(plan, false);  // its finish call draws
}

SPEC_EXPORT int spec_verify_sample_finish(const void *target_logits, const void *draft_logits,
                                          const int32_t *draft_tokens, const float *uniforms,
                                          int B, int k, int V, float temperature, float top_p,
                                          int mode, int dtype, int32_t *out_tokens,
                                          int32_t *out_num_accepted, void *workspace,
                                          size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    const int rc = plan_chain(target_logits, draft_logits, draft_tokens, uniforms, B, k, V,
                              temperature, top_p, mode, dtype, out_tokens, out_num_accepted,
                              workspace, workspace_bytes, stream, &plan);
    if (rc != SPEC_OK || B == 0) return rc;
    return launch_chain_finish(plan);
}

SPEC_EXPORT int spec_verify_sample_probs(const void *target_logits, const float *draft_probs,
                                         const int32_t *draft_tokens, const float *uniforms,
                                         int B, int k, int V, float temperature, float top_p,
                                         int top_k, int dtype, int32_t *out_tokens,
                                         int32_t *out_num_accepted, void *workspace,
                                         size_t workspace_bytes, spec_stream_t stream) {
    ChainPlan plan;
    int rc = plan_chain(target_logits, draft_probs, draft_tokens, uniforms, B, k, V, temperature,
                        top_p, SPEC_STOCHASTIC, dtype, out_tokens, out_num_accepted, workspace,
                        workspace_bytes, stream, &plan, true, top_k);
    if (rc != SPEC_OK || B == 0) return rc;
    rc = launch_chain_rows(plan, true);
    if (rc != SPEC_OK) return rc;
    return launch_chain_finish(plan);
}

SPEC_EXPORT int spec_verify_tree(const void *target_logits, const int32_t *parents,
                                 const int32_t *node_tokens, int B, int N, int V, int D,
                                 int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                                 int32_t *out_path, void *workspace, size_t workspace_bytes,
                                 spec_stream_t stream) {
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
    if (!tree_sizes_ok(B, N, V) || D < 0 || D >= N) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;  // nothing is read or written: any pointer will do
    if (!target_logits || !parents || !node_tokens || !out_tokens || !out_num_accepted ||
        !workspace)
        return SPEC_ERR_NULL;
    const size_t esz = dtype == SPEC_F32 ? 4 : 2;
    if (!aligned(target_logits, esz) || !aligned(parents, 4) || !aligned(node_tokens, 4) ||
        !aligned(out_tokens, 4) || !aligned(out_num_accepted, 4) ||
        (out_path && !aligned(out_path, 4)) || !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < carve(nullptr, B, N, V, nullptr, false, false)) return SPEC_ERR_WORKSPACE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Workspace ws;
    carve(workspace, B, N, V, &ws, false, false);
    RowView rv;
    rv.target = target_logits;
    rv.draft = nullptr;
    rv.V = V;
    rv.k = 0;
    rv.R = N;
    rv.draft_rows_from = N;
    rv.tgt_rows_per_seq = N;
    SeqArgs sq = {};
    sq.work = kSeqNone;
    const int rc = launch_stream_rows(rv, sq, B * N, 1.4426950408889634f, ws, 1, dtype, st);
    if (rc != SPEC_OK) return rc;
    TreeArgs ta;
    ta.parents = parents;
    ta.node_tokens = node_tokens;
    ta.B = B;
    ta.N = N;
    ta.V = V;
    ta.D = D;
    ta.out_tokens = out_tokens;
    ta.out_num = out_num_accepted;
    ta.out_path = out_path;
    ta.ws = ws;
    return launch_tree(ta, st);
}

SPEC_EXPORT int spec_verify_tree_sample_workspace_size(int B, int N, int V, size_t *bytes) {
    if (!bytes) return SPEC_ERR_NULL;
    if (!tree_sizes_ok(B, 2 * N, V) || N > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
    *bytes = carve(nullptr, B, 2 * N, V, nullptr, false, true);
    return SPEC_OK;
}

SPEC_EXPORT int spec_verify_tree_sample(const void *target_logits, const void *draft_logits,
                                        const int32_t *parents, const int32_t *node_tokens,
                                        const float *uniforms, int B, int N, int V, int D,
                                        float temperature, float top_p, int top_k, int dtype,
                                        int32_t *out_tokens, int32_t *out_num_accepted,
                                        int32_t *out_path, void *workspace,
                                        size_t workspace_bytes, spec_stream_t stream) {
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
    if (N < 1 || N > SPEC_MAX_TREE_NODES || !tree_sizes_ok(B, 2 * N, V) || D < 0 || D >= N)
        return SPEC_ERR_SHAPE;
    if (!(temperature > 0.0f) || !std::isfinite(temperature) || !(top_p > 0.0f) ||
        !(top_p <= 1.0f))
        return SPEC_ERR_PARAM;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits || !parents || !node_tokens || !uniforms ||
        !out_tokens || !out_num_accepted || !workspace)
        return SPEC_ERR_NULL;
    const size_t esz = dtype == SPEC_F32 ? 4 : 2;
    if (!aligned(target_logits, esz) || !aligned(draft_logits, esz) || !aligned(parents, 4) ||
        !aligned(node_tokens, 4) || !aligned(uniforms, 4) || !aligned(out_tokens, 4) ||
        !aligned(out_num_accepted, 4) || (out_path && !aligned(out_path, 4)) ||
        !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < carve(nullptr, B, 2 * N, V, nullptr, false, true)) return SPEC_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Workspace ws;
    carve(workspace, B, 2 * N, V, &ws, false, true);
    const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    // Row statistics of the 2N rows of every sequence (targets, then drafts).
    RowView rv;
    rv.target = target_logits;
    rv.draft = draft_logits;
    rv.V = V;
    rv.k = N;
    rv.R = 2 * N;
    rv.draft_rows_from = N;
    rv.tgt_rows_per_seq = N;
    SeqArgs sq = {};
    sq.work = kSeqNone;
    const int kk = top_k > 0 && top_k < V ? top_k : 0;
    int rc;
    if (top_p < 1.0f || kk > 0) {
        ToppArgs ta;
        ta.rows = rv;
        ta.seq = sq;
        ta.c = c;
        ta.temperature = temperature;
        ta.top_p = top_p;
        ta.top_k = kk;
        ta.ws = ws;
        rc = launch_topp_rows(ta, B * 2 * N, dtype, st);
    } else {
        rc = launch_stream_rows(rv, sq, B * 2 * N, c, ws, 0, dtype, st);
    }
    if (rc != SPEC_OK) return rc;
    TreeSampleArgs a;
    a.target = target_logits;
    a.draft = draft_logits;
    a.parents = parents;
    a.node_tokens = node_tokens;
    a.uniforms = uniforms;
    a.B = B;
    a.N = N;
    a.V = V;
    a.D = D;
    a.c = c;
    a.out_tokens = out_tokens;
    a.out_num = out_num_accepted;
    a.out_path = out_path;
    a.ws = ws;
    return launch_tree_sample(a, dtype, st);
}

SPEC_EXPORT int spec_verify_tree_mask(const int32_t *parents, const int32_t *pos0, int B, int N,
                                      uint8_t *out_mask, float *out_bias, int32_t *out_pos,
                                      spec_stream_t stream) {
    if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES ||
        static_cast<long long>(B) * ((N + 31) / 32) > INT_MAX)
        return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;
    if (!parents) return SPEC_ERR_NULL;
    if (!aligned(parents, 4) || (pos0 && !aligned(pos0, 4)) || (out_bias && !aligned(out_bias, 4)) ||
        (out_pos && !aligned(out_pos, 4)))
        return SPEC_ERR_ALIGN;
    if (!out_mask && !out_bias && !out_pos) return SPEC_OK;
    TreeMaskArgs a;
    a.parents = parents;
    a.pos0 = pos0;
    a.B = B;
    a.N = N;
    a.mask = out_mask;
    a.bias = out_bias;
    a.pos = out_pos;
    return launch_tree_mask(a, reinterpret_cast<cudaStream_t>(stream));
}

SPEC_EXPORT int spec_verify_last_error(void *workspace, size_t workspace_bytes,
                                       spec_stream_t stream) {
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

SPEC_EXPORT int spec_verify_intermediates(const void *workspace, size_t workspace_bytes, int B,
                                          int k, int V, float *P, float *Q, float *Z, float *S,
                                          spec_stream_t stream) {
    if (!workspace) return SPEC_ERR_NULL;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    if (workspace_bytes < carve(nullptr, B, 2 * k + 1, V, nullptr, true, false))
        return SPEC_ERR_WORKSPACE;
    if (B == 0) return SPEC_OK;
    Workspace ws;
    carve(const_cast<void *>(workspace), B, 2 * k + 1, V, &ws, true, false);
    return launch_intermediates(ws, B, k, P, Q, Z, S, reinterpret_cast<cudaStream_t>(stream));
}

SPEC_EXPORT int spec_verify_acceptance(const void *target_logits, const void *draft_logits, int B,
                                       int k, int V, float temperature, float top_p, int top_k,
                                       int dtype,
                                       float *out_beta, float *out_tv, void *workspace,
                                       size_t workspace_bytes, spec_stream_t stream) {
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
    if (!chain_sizes_ok(B, k, V)) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits || !out_beta || !workspace) return SPEC_ERR_NULL;
    if (!(temperature > 0.0f) || !std::isfinite(temperature) || !(top_p > 0.0f) ||
        !(top_p <= 1.0f))
        return SPEC_ERR_PARAM;
    const size_t esz = dtype == SPEC_F32 ? 4 : 2;
    if (!aligned(target_logits, esz) || !aligned(draft_logits, esz) || !aligned(out_beta, 4) ||
        (out_tv && !aligned(out_tv, 4)) || !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    const bool topk_on = top_k > 0 && top_k < V;
    if (workspace_bytes < carve(nullptr, B, 2 * k + 1, V, nullptr, true, topk_on))
        return SPEC_ERR_WORKSPACE;
    AcceptArgs a;
    carve(workspace, B, 2 * k + 1, V, &a.ws, true, topk_on);
    a.rows.target = target_logits;
    a.rows.draft = draft_logits;
    a.rows.V = V;
    a.rows.k = k;
    a.rows.R = 2 * k + 1;
    a.rows.draft_rows_from = k + 1;
    a.rows.tgt_rows_per_seq = k + 1;
    a.pairs = static_cast<long long>(B) * k;
    a.total = a.pairs * V;
    a.seg = 0;
    a.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    const bool masked = top_p < 1.0f || (top_k > 0 && top_k < V);
    a.list = masked ? 1 : 0;
    a.beta = out_beta;
    a.tv = out_tv;
    return launch_accept(a, dtype, masked, reinterpret_cast<cudaStream_t>(stream));
}

SPEC_EXPORT const char *spec_verify_status_string(int status) {
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
    case SPEC_DATA_TREE_SHAPE:
        return "parents is not a rooted tree in topological order within depth D";
    case SPEC_DATA_PROB_RANGE: return "a gathered draft probability lies outside [0, 1]";
    default: return "unknown status";
    }
}
