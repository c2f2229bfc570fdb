// select.cu -- the top-p / top-k threshold of every row, one warp per row.
//
// The thresholds are defined in topp.cu's header ("3.5 Speculative
// Decoding", "Notation"; top-k: "246 Speculative Decoding", 6): lam is the
// largest key whose fixed-point mass from the top reaches top_p Z (ties of
// lam kept), tau the K-th largest key by count.  Both are step functions
// of the key with exact integer weights, so a value histogram (monotone
// bins) followed by a bisection over the keys of the crossing bin finds
// exactly the key the histogram select of topp.cu finds.
//
// select_warp_kernel  one warp per row, no block barriers, one wave:
//   1. the row's summary (rows.cu) names the groups whose max reaches the
//      floor F -- m - kToppTry T, or with top-k a lower bound of the K-th
//      largest logit (the K-th largest of the group maxima each lane kept)
//      -- and only those vectors are read again (mostly one per group);
//   2. tau (count) and lam (mass) over the gathered logits: a 256-bin value
//      histogram, then a bisection inside the crossing bin;
//   3. for a target row, its nucleus list ranked by index with the draft
//      value at each index;
//   4. the row record, and the sequence's decision when this was its last
//      row.
// A row this path cannot take (more than kSwList logits or kSwGroups
// groups >= F, a nucleus that reaches below F, more than 32 pieces, K >
// kSwMaxK) is marked in ws.defer and taken by topp_kernel, launched next,
// whose other CTAs exit.  (A nucleus list longer than kNucCap is left to
// the final kernel, as topp_kernel leaves it.)

#include "stream.cuh"

namespace specv {
namespace {

constexpr int kSwWarps = 2;      // rows (warps) per CTA
constexpr int kSwList = 2048;    // gathered logits one warp holds
constexpr int kSwGroups = 2048;  // selected groups one warp lists
constexpr int kSwMaxK = 128;     // largest top-k the warp path takes
constexpr int kSwTop = 8;        // group keys each lane keeps for the top-k bound
constexpr int kSwBuckets = 256;  // index buckets of the nucleus ranking
constexpr int kSwBins = 256;     // value bins of the threshold select
static_assert(kNucCap * 2 <= kSwGroups, "the nucleus (index, logit) pairs reuse gl");
static_assert(kSwBuckets + kNucCap <= kSwList, "the ranking scratch reuses lx");

struct SwWarp {
    float lv[kSwList];      // gathered logits
    int lx[kSwList];        // ... and their indices in the row
    uint32_t gl[kSwGroups]; // selected groups: u1 << 25 | all << 24 | entry (in the row);
                            // then the crossing bin's logits; then the nucleus,
                            // (index, logit bits) pairs
    unsigned long long hist[kSwBins];  // the threshold select's histogram
    int pc_off[33], pc_a0[32], pc_nv[32];  // the row's pieces: summary offset, vectors
};
struct SwShared {
    SwWarp w[kSwWarps];
};

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Exclusive warp prefix of cnt (lane order) and the total.
__device__ __forceinline__ int warp_excl(int cnt, int &tot) {
    const int lane = threadIdx.x & 31;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    return incl - cnt;
}

// Append this lane's logits h[e] with bit e of `mask` set (indices x0 + e)
// to the warp's list of n (warp-uniform; counted past kSwList: overflow).
// Every lane of the warp calls it.
template <int N>
__device__ __forceinline__ void sw_push(SwWarp &sw, int &n, uint32_t mask, const float (&h)[N],
                                        int x0) {
    int tot;
    int p = n + warp_excl(__popc(mask), tot);
#pragma unroll
    for (int e = 0; e < N; ++e)
        if (mask & (1u << e)) {
            if (p < kSwList) {
                sw.lv[p] = h[e];
                sw.lx[p] = x0 + e;
            }
            ++p;
        }
    n += tot;
}

template <typename T, bool TOPK>
__global__ void __launch_bounds__(kSwWarps * 32) select_warp_kernel(const ToppArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(16) unsigned char sw_smem[];
    constexpr int P = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    SwWarp &sw = reinterpret_cast<SwShared *>(sw_smem)->w[wid];
    const int row = blockIdx.x * kSwWarps + wid;
    // The statistics grid's records and summaries: visible once it has
    // completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (row >= a.rows_total) return;  // whole warp
    const int V = a.rows.V;
    const float c = a.c, tryT = kToppTry * a.temperature;
    const T *rowp = row_ptr<T>(a.rows, row);
    RowRec *rec = a.ws.rows + row;
    const float m = __ldcg(&rec->m), Z = __ldcg(&rec->z_full);
    const uint32_t flags = __ldcg(&rec->flags);
    const int R = a.rows.R, kk = a.rows.k;
    const int bq = row / R, rq = row - bq * R;
    const bool nuc_row = a.seq.list_draw && rq <= kk;
    const int tr = bq * (kk + 1) + rq;
    auto defer = [&]() {
        if (lane == 0) a.ws.defer[row] = 1u;
    };
    uint32_t lam = 0u;
    float zk = Z;
    if (flags == 0u) {
        // ---- the row's pieces: lane i < np holds piece i
        const long long rbase = static_cast<long long>(row) * V;
        const long long wf = rbase / a.seg, wl = (rbase + V - 1) / a.seg;
        const int np = static_cast<int>(wl - wf + 1);
        if (np > 32) return defer();
        int p_lo = 0, p_hi = 0, p_a0 = 0, p_nv = 0, p_ng = 0;
        if (lane < np) {
            piece_bounds(row, V, a.seg, wf + lane, p_lo, p_hi);
            const Span<T> sp(rowp, p_lo, p_hi);
            p_a0 = sp.a0;
            p_nv = sp.nvec;
            p_ng = (sp.nvec + kGroupVecs - 1) / kGroupVecs * 32;
        }
        int ng_tot;
        const int p_off = warp_excl(p_ng, ng_tot);
        if ((ng_tot >> 24) != 0) return defer();
        if (lane < np) {
            sw.pc_off[lane] = p_off;
            sw.pc_a0[lane] = p_a0;
            sw.pc_nv[lane] = p_nv;
        }
        if (lane == 0) sw.pc_off[np] = ng_tot;
        __syncwarp();
        auto piece_of = [&](int e) {
            int i = 0;
            while (i + 1 < np && sw.pc_off[i + 1] <= e) ++i;
            return i;
        };
        const uint32_t *sum = a.ws.sum + static_cast<size_t>(row) * a.ws.sum_stride;
        // Every summary entry of the row (index e among the row's entries):
        // f(e, entry, valid), every lane the same number of times; four
        // entries per 16-byte load, eight loads in flight per lane.  (Piece
        // offsets are multiples of 32 entries and rows start 128-byte
        // aligned.)
        auto for_entries = [&](auto &&f) {
            const uint4 *src = reinterpret_cast<const uint4 *>(sum);
            const int nv4 = ng_tot / 4;
            constexpr int kU = 8;
            for (int base = 0; base < nv4; base += 32 * kU) {  // uniform
                uint4 w[kU];
#pragma unroll
                for (int r = 0; r < kU; ++r) {
                    const int v = base + r * 32 + lane;
                    w[r] = v < nv4 ? __ldcg(src + v) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int r = 0; r < kU; ++r) {
                    const int v = base + r * 32 + lane;
                    const bool ok = v < nv4;
                    f(4 * v, w[r].x, ok);
                    f(4 * v + 1, w[r].y, ok);
                    f(4 * v + 2, w[r].z, ok);
                    f(4 * v + 3, w[r].w, ok);
                }
            }
        };
        // A selected group's descriptor: its vector of the max, whether the
        // rest must be read too, its entry index.
        auto desc = [&](int e, uint32_t en, float floor) {
            return (static_cast<uint32_t>(entry_vec(en)) << 25) |
                   (entry_rest(en) >= floor ? 1u << 24 : 0u) | static_cast<uint32_t>(e);
        };
        const uint32_t kneg = sum_key(kNegInf);
        const bool topk = TOPK && a.top_k > 0 && a.top_k < V;
        float F = __fsub_rn(m, tryT);
        int ngr = 0;
        bool listed = false;  // the group list is built
        if (topk) {
            // ---- a lower bound of the K-th largest logit: each lane keeps
            // its kSwTop largest group entries; the K-th largest of their
            // keys.  Unless some lane kept kSwTop entries above the bound
            // (then it may have dropped more), those entries are the groups
            // to read.
            if (a.top_k > kSwMaxK) return defer();
            uint32_t tk[kSwTop], te[kSwTop], tp[kSwTop];  // key, entry, index
#pragma unroll
            for (int t = 0; t < kSwTop; ++t) tk[t] = te[t] = tp[t] = 0u;
            for_entries([&](int e, uint32_t en, bool ok) {
                uint32_t k = ok ? en >> 16 : 0u;
                if (k <= kneg || k <= tk[kSwTop - 1]) return;
                uint32_t xe = en, xp = static_cast<uint32_t>(e);
#pragma unroll
                for (int t = 0; t < kSwTop; ++t)  // insert, descending
                    if (k > tk[t]) {
                        const uint32_t a1 = tk[t], a2 = te[t], a3 = tp[t];
                        tk[t] = k;
                        te[t] = xe;
                        tp[t] = xp;
                        k = a1;
                        xe = a2;
                        xp = a3;
                    }
            });
            auto count_ge = [&](uint32_t k) {
                unsigned int c2 = 0u;
#pragma unroll
                for (int t = 0; t < kSwTop; ++t) c2 += tk[t] >= k;
                return __reduce_add_sync(0xFFFFFFFFu, c2);
            };
            const unsigned int K = static_cast<unsigned int>(a.top_k);
            uint32_t lo = kneg + 1u, hi = 0xFFFFu;
            if (count_ge(lo) < K) return defer();
            while (lo < hi) {
                const uint32_t mid = (lo + hi + 1u) >> 1;
                if (count_ge(mid) >= K) lo = mid;
                else hi = mid - 1u;
            }
            const uint32_t kb = sizeof(T) == 4 ? lo - 1u : lo;  // fp32: one bf16 step below
            if (kb <= kneg) return defer();
            F = sum_value(kb);
            if (!__any_sync(0xFFFFFFFFu, tk[kSwTop - 1] >= kb)) {
#pragma unroll
                for (int t = 0; t < kSwTop; ++t) {
                    const bool want = tk[t] >= kb;  // (a group max is its key's value)
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, want);
                    const int pos = ngr + __popc(bal & ((1u << lane) - 1u));
                    if (want && pos < kSwGroups) sw.gl[pos] = desc(static_cast<int>(tp[t]), te[t], F);
                    ngr += __popc(bal);
                }
                listed = true;
            }
        }
        // ---- the groups whose max reaches F, listed
        if (!listed)
            for_entries([&](int e, uint32_t en, bool ok) {
                const bool want = ok && entry_max(en) >= F;
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, want);
                const int pos = ngr + __popc(bal & ((1u << lane) - 1u));
                if (want && pos < kSwGroups) sw.gl[pos] = desc(e, en, F);
                ngr += __popc(bal);
            });
        if (ngr > kSwGroups) return defer();
        __syncwarp();
        // ---- their vectors (the max's; all four where the rest's bound
        // reaches F) and the pieces' ragged ends, into the list
        int n = 0;
        {
            // ragged ends: at most P - 1 logits before a0 and after a1 per
            // piece; kR per lane and round, loaded together
            constexpr int kR = 4;
            const int nr = np * 2 * (P - 1);
            for (int base = 0; base < nr; base += 32 * kR) {  // uniform
                float h[kR];
                int x[kR];
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int t = base + r * 32 + lane;
                    const int i = t / (2 * (P - 1)), j = t - i * 2 * (P - 1);
                    x[r] = -1;
                    h[r] = kNegInf;
                    if (t < nr) {
                        const int a0 = sw.pc_a0[i], a1 = a0 + sw.pc_nv[i] * P;
                        int lo, hi;
                        piece_bounds(row, V, a.seg, wf + i, lo, hi);
                        const int xx = j < P - 1 ? lo + j : a1 + (j - (P - 1));
                        if (j < P - 1 ? xx < a0 : xx < hi) {
                            x[r] = xx;
                            h[r] = to_f32(rowp[xx]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const float hv[1] = {h[r]};
                    sw_push(sw, n, x[r] >= 0 && h[r] >= F ? 1u : 0u, hv, x[r]);
                }
            }
        }
        constexpr int kG = 4;  // groups per lane and round
        for (int g0 = 0; g0 < ngr; g0 += 32 * kG) {  // uniform
            uint4 q[kG];
            int gx[kG], ga[kG], gv[kG], gb[kG];
            bool rest[kG];
#pragma unroll
            for (int r = 0; r < kG; ++r) {
                const int g = g0 + r * 32 + lane;
                const bool has = g < ngr;
                const uint32_t d = has ? sw.gl[g] : 0u;
                const int e = static_cast<int>(d & 0xFFFFFFu), u1 = static_cast<int>((d >> 25) & 3u);
                const int i = has ? piece_of(e) : 0;
                const int a0 = sw.pc_a0[i], nv = sw.pc_nv[i];
                const int j = e - sw.pc_off[i];
                const int bl = (j >> 5) * kGroupVecs + (j & 31);  // the group's first vector
                const int v = bl + u1 * 32;
                gx[r] = a0 + v * P;
                q[r] = has && v < nv ? __ldcg(reinterpret_cast<const uint4 *>(rowp + a0) + v)
                                     : neg_inf_vec<T>();
                rest[r] = has && ((d >> 24) & 1u);
                ga[r] = a0;
                gv[r] = nv;
                gb[r] = bl | (u1 << 29);
            }
#pragma unroll
            for (int r = 0; r < kG; ++r) {
                float h[P];
                unpack<T>(q[r], h);
                uint32_t mask = 0u;
#pragma unroll
                for (int e = 0; e < P; ++e)
                    if (h[e] >= F) mask |= 1u << e;
                sw_push(sw, n, mask, h, gx[r]);
            }
            // groups whose other vectors may reach F: those vectors too (rare)
#pragma unroll
            for (int r = 0; r < kG; ++r) {
                if (!__any_sync(0xFFFFFFFFu, rest[r])) continue;  // uniform
                const int bl = gb[r] & 0x1FFFFFFF, u1 = gb[r] >> 29;
                uint4 qq[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int v = bl + u * 32;
                    qq[u] = rest[r] && u != u1 && v < gv[r]
                                ? __ldcg(reinterpret_cast<const uint4 *>(rowp + ga[r]) + v)
                                : neg_inf_vec<T>();
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    float h[P];
                    unpack<T>(qq[u], h);
                    uint32_t mask = 0u;
#pragma unroll
                    for (int e = 0; e < P; ++e)
                        if (h[e] >= F) mask |= 1u << e;
                    sw_push(sw, n, mask, h, ga[r] + (bl + u * 32) * P);
                }
            }
        }
        if (n > kSwList) return defer();
        __syncwarp();
        // ---- the thresholds: a histogram of the gathered logits by value,
        // then exact among the crossing bin's logits
        const float negmc = -__fmul_rn(m, c);
        auto mass = [&](float l) {
            return __float2ull_rn(__fmul_rn(ex2(__fmaf_rn(l, c, negmc)), kFix));
        };
        auto kval = [&](uint32_t k) { return key_float(sizeof(T) == 2 ? k << 16 : k); };
        uint32_t kmin = 0xFFFFFFFFu;
        for (int i = lane; i < n; i += 32) kmin = min(kmin, okey<T>(sw.lv[i]));
        kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
        // Total weight (count or mass) of the gathered logits with key >= k.
        auto weight_ge = [&](bool count, uint32_t k) {
            unsigned long long s = 0ull;
            for (int i = lane; i < n; i += 32) {
                const float l = sw.lv[i];
                if (okey<T>(l) >= k) s += count ? 1ull : mass(l);
            }
            return warp_sum_u64(s);
        };
        // The largest key k >= kfl whose weight over the gathered logits
        // with key >= k reaches target (0xFFFFFFFF if none); *wk gets it.
        // A histogram of kSwBins bins uniform in value over [value(kfl), m]
        // -- bins are monotone in the logit, so the bin where the weight
        // from the top first reaches target holds the answer -- then a
        // bisection over the keys of that bin's logits alone (gathered
        // into gl's scratch).
        auto select = [&](bool count, uint32_t kfl, unsigned long long target,
                          unsigned long long &wk) -> uint32_t {
            const float span = __fsub_rn(m, kval(kfl));
            const float inv = span > 0.0f ? static_cast<float>(kSwBins) / span : 0.0f;
            auto vbin = [&](float l) {
                return min(static_cast<int>(__fmul_rn(__fsub_rn(m, l), inv)), kSwBins - 1);
            };
            for (int t = lane; t < kSwBins; t += 32) sw.hist[t] = 0ull;
            __syncwarp();
            for (int i = lane; i < n; i += 32) {
                const float l = sw.lv[i];
                if (okey<T>(l) >= kfl) atomicAdd(&sw.hist[vbin(l)], count ? 1ull : mass(l));
            }
            __syncwarp();
            constexpr int kPer = kSwBins / 32;  // lane L owns bins kPer L .. kPer L + kPer - 1
            unsigned long long h[kPer], tot = 0ull;
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                h[t] = sw.hist[kPer * lane + t];
                tot += h[t];
            }
            unsigned long long incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= target);
            if (!hit) return 0xFFFFFFFFu;
            const int src = __ffs(hit) - 1;
            int b0 = 0;
            unsigned long long above = incl - tot;
            if (lane == src) {
                int t = 0;
                while (above + h[t] < target) above += h[t++];
                b0 = kPer * lane + t;
            }
            b0 = __shfl_sync(0xFFFFFFFFu, b0, src);
            above = __shfl_sync(0xFFFFFFFFu, above, src);
            // the crossing bin's logits
            float *bv = reinterpret_cast<float *>(sw.gl);
            int nb = 0;
            uint32_t klo = 0xFFFFFFFFu, khi = 0u;
            for (int i0 = 0; i0 < n; i0 += 32) {  // uniform
                const int i = i0 + lane;
                const float l = i < n ? sw.lv[i] : kNegInf;
                const bool in = i < n && okey<T>(l) >= kfl && vbin(l) == b0;
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
                if (in) {
                    bv[nb + __popc(bal & ((1u << lane) - 1u))] = l;
                    klo = min(klo, okey<T>(l));
                    khi = max(khi, okey<T>(l));
                }
                nb += __popc(bal);
            }
            klo = __reduce_min_sync(0xFFFFFFFFu, klo);
            khi = __reduce_max_sync(0xFFFFFFFFu, khi);
            __syncwarp();
            auto bin_ge = [&](uint32_t k) {
                unsigned long long s2 = 0ull;
                for (int i = lane; i < nb; i += 32) {
                    const float l = bv[i];
                    if (okey<T>(l) >= k) s2 += count ? 1ull : mass(l);
                }
                return above + warp_sum_u64(s2);
            };
            uint32_t lo = klo, hi = khi;
            while (lo < hi) {
                const uint32_t mid = lo + (hi - lo + 1u) / 2u;
                if (bin_ge(mid) >= target) lo = mid;
                else hi = mid - 1u;
            }
            wk = bin_ge(lo);
            __syncwarp();
            return lo;
        };
        uint32_t kfloor = kmin;  // the kept set's smallest key
        float zsel = Z;
        bool have_lam = false;
        if (topk) {
            // tau: the largest key with count >= K (the list holds >= K logits)
            unsigned long long cnt;
            const uint32_t tau =
                select(true, kmin, static_cast<unsigned long long>(a.top_k), cnt);
            if (tau == 0xFFFFFFFFu) return defer();
            kfloor = tau;
            zsel = __fmul_rn(__ull2float_rn(weight_ge(false, tau)), 1.0f / kFix);
            if (!(a.top_p < 1.0f)) {
                lam = tau;
                zk = zsel;
                have_lam = true;
            }
        }
        if (!have_lam) {
            // lam: the largest key >= kfloor whose mass from the top reaches
            // top_p zsel; if the gathered mass falls short, the nucleus
            // reaches below F: topp_kernel reads the row.
            const unsigned long long tgt =
                __float2ull_rn(__fmul_rn(__fmul_rn(a.top_p, zsel), kFix));
            unsigned long long wl2;
            lam = select(false, kfloor, tgt, wl2);
            if (lam == 0xFFFFFFFFu) return defer();
            zk = __fmul_rn(__ull2float_rn(wl2), 1.0f / kFix);
        }
        // ---- the nucleus list of a target row for the final draw
        if (nuc_row) {
            uint2 *nuc = reinterpret_cast<uint2 *>(sw.gl);  // (index, logit bits)
            int nn = 0;
            for (int i0 = 0; i0 < n; i0 += 32) {  // uniform
                const int i = i0 + lane;
                const bool keep = i < n && okey<T>(sw.lv[i]) >= lam;
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
                const int pos = nn + __popc(bal & ((1u << lane) - 1u));
                if (keep && pos < kNucCap)
                    nuc[pos] = make_uint2(static_cast<uint32_t>(sw.lx[i]), __float_as_uint(sw.lv[i]));
                nn += __popc(bal);
            }
            __syncwarp();
            const bool ok = nn <= kNucCap;
            if (ok) {
                // Rank by index: bucket the entries by index (kSwBuckets
                // buckets over [0, V)), scan the counts, place each entry
                // in its bucket, then count the smaller indices inside its
                // bucket alone.  Scratch: the list's index array.
                int *cnt = sw.lx, *byb = sw.lx + kSwBuckets;
                for (int t = lane; t < kSwBuckets; t += 32) cnt[t] = 0;
                __syncwarp();
                auto bucket = [&](uint32_t x) {
                    return static_cast<int>((static_cast<long long>(x) * kSwBuckets) / V);
                };
                for (int i = lane; i < nn; i += 32) atomicAdd(&cnt[bucket(nuc[i].x)], 1);
                __syncwarp();
                constexpr int kPer = kSwBuckets / 32;
                int c8[kPer], tot8 = 0;
#pragma unroll
                for (int t = 0; t < kPer; ++t) {
                    c8[t] = cnt[lane * kPer + t];
                    tot8 += c8[t];
                }
                int n_all;
                int st = warp_excl(tot8, n_all);
                __syncwarp();
#pragma unroll
                for (int t = 0; t < kPer; ++t) {  // cnt becomes each bucket's start
                    cnt[lane * kPer + t] = st;
                    st += c8[t];
                }
                __syncwarp();
                // Place: cnt[bk], the bucket's start, is its cursor.
                for (int i = lane; i < nn; i += 32) {
                    const int bk = bucket(nuc[i].x);
                    const int slot = atomicAdd(&cnt[bk], 1);
                    byb[slot] = static_cast<int>(nuc[i].x);
                }
                __syncwarp();
                // cnt[bk] is now the end of bucket bk; its start is the end
                // of bucket bk - 1 (0 for the first)
                uint4 *L = a.ws.nuc + static_cast<size_t>(tr) * kNucCap;
                const size_t doff = (static_cast<size_t>(bq) * kk + rq) * V;
                const T *drow = rq < kk && !a.seq.qprob
                                    ? static_cast<const T *>(a.rows.draft) + doff
                                    : nullptr;
                const float *dprob = rq < kk && a.seq.qprob
                                         ? static_cast<const float *>(a.rows.draft) + doff
                                         : nullptr;
                constexpr int kQ = 8;  // draft values loaded together per lane
                for (int i0 = lane; i0 < nn; i0 += 32 * kQ) {
                    float lq[kQ];
#pragma unroll
                    for (int r = 0; r < kQ; ++r) {
                        const int i = i0 + r * 32;
                        const uint32_t x = i < nn ? nuc[i].x : 0u;
                        lq[r] = i >= nn ? 0.0f
                                : drow  ? to_f32(drow[x])
                                : dprob ? dprob[x]
                                        : 0.0f;
                    }
#pragma unroll
                    for (int r = 0; r < kQ; ++r) {
                        const int i = i0 + r * 32;
                        if (i >= nn) break;
                        const uint2 en = nuc[i];
                        const int bk = bucket(en.x);
                        const int s0 = bk ? cnt[bk - 1] : 0, s1 = cnt[bk];
                        int rank = s0;
                        for (int j = s0; j < s1; ++j) rank += static_cast<uint32_t>(byb[j]) < en.x;
                        L[rank] = make_uint4(en.x, en.y, __float_as_uint(lq[r]), 0u);
                    }
                }
            }
            if (lane == 0) a.ws.nuc_n[tr] = ok ? nn : -1;
        }
    } else if (nuc_row && lane == 0) {
        a.ws.nuc_n[tr] = -1;
    }
    if (lane == 0) {
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
    __threadfence();  // the record and nucleus list, for whichever warp decides the sequence
    __syncwarp();
    row_done<T>(a.rows, a.seq, a.ws, a.c, row);
}

template <typename K>
bool sw_smem_ok(K kernel, int slot) {
    constexpr int kMaxDev = 64;
    static int done[kMaxDev][4];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    if (__atomic_load_n(&done[dev][slot], __ATOMIC_RELAXED)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sizeof(SwShared)) != cudaSuccess)
        return false;
    __atomic_store_n(&done[dev][slot], 1, __ATOMIC_RELAXED);
    return true;
}

template <typename T, bool TOPK>
int launch_select_warp_t(const ToppArgs &a, cudaStream_t st) {
    auto kernel = select_warp_kernel<T, TOPK>;
    if (!sw_smem_ok(kernel, (sizeof(T) == 2 ? 1 : 0) + (TOPK ? 2 : 0))) return SPEC_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.rows_total + kSwWarps - 1) / kSwWarps));
    cfg.blockDim = dim3(kSwWarps * 32);
    cfg.dynamicSmemBytes = sizeof(SwShared);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

int launch_select_warp(const ToppArgs &a, int dtype, cudaStream_t st) {
    const bool topk = a.top_k > 0;
    if (dtype == SPEC_F32)
        return topk ? launch_select_warp_t<float, true>(a, st)
                    : launch_select_warp_t<float, false>(a, st);
    return topk ? launch_select_warp_t<uint16_t, true>(a, st)
                : launch_select_warp_t<uint16_t, false>(a, st);
}

}  // namespace specv
