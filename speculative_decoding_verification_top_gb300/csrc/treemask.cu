// treemask.cu -- tree attention inputs for B candidate trees: the step
// just before the target pass whose logits spec_verify_tree reads.
//
// "3.5 Speculative Decoding" (llm-learning-path), "Tree verification": the
// flattened tree is scored in one target pass in which every node attends
// to the context and to its own ancestors only (not to siblings), and nodes
// at the same depth receive the same position index (for RoPE).
// "Speculative Decoding: Mathematical Foundations, ..." (llms.blog),
// "Tree-Based Verification and Custom Attention Masks": the mask as an
// additive bias, M_ij = 0 where node j is an ancestor of node i, -inf
// elsewhere.
//
// tree_mask_kernel   one CTA per (tree, block of rows): it stages its
//                    tree's parent array in shared memory and checks it;
//                    each warp takes up to 32 rows (fewer for small batches),
//                    its lanes walk those ancestor chains at once into
//                    per-row shared bitsets (parents[n] < n, so each walk
//                    ends at the root), then the warp writes the rows one
//                    after another, coalesced, with
//                    16-byte stores when a row is 16-byte aligned.  The
//                    output is write-bound: B N N bytes (mask), 4 B N N
//                    (bias).

#include "common.cuh"

namespace specv {
namespace {

constexpr int kTmWords = SPEC_MAX_TREE_NODES / 32;

// Four mask bits (bit 0 first) as four bytes of 0 / 1, little-endian.
__device__ __forceinline__ uint32_t bits_to_bytes(uint32_t b4) {
    return (b4 & 1u) | ((b4 >> 1) & 1u) << 8 | ((b4 >> 2) & 1u) << 16 | ((b4 >> 3) & 1u) << 24;
}

struct TreeMaskShared {
    int par[SPEC_MAX_TREE_NODES];
    uint32_t bits[kWarps][32][kTmWords + 1];  // a bitset per row (+1: bank spread)
    int bad;
};

__global__ void __launch_bounds__(kThreads) tree_mask_kernel(const TreeMaskArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TreeMaskShared &sh = *reinterpret_cast<TreeMaskShared *>(smem_raw);
    const int N = a.N, RW = a.rows_per_warp, cta_rows = kWarps * RW;
    const int nrb = (N + cta_rows - 1) / cta_rows;
    const int b = blockIdx.x / nrb, rblock = blockIdx.x - b * nrb;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) sh.bad = 0;
    __syncthreads();
    const int32_t *par = a.parents + static_cast<size_t>(b) * N;
    bool bad = false;
    for (int n = tid; n < N; n += kThreads) {
        const int p = par[n];
        sh.par[n] = p;
        if (n == 0 ? p != -1 : (p < 0 || p >= n)) bad = true;
    }
    if (bad) sh.bad = 1;
    __syncthreads();
    const bool ok = sh.bad == 0;
    const int words = (N + 31) / 32;
    const int r0 = rblock * cta_rows + warp * RW;  // this warp's RW rows
    if (r0 >= N) return;
    const int nr = min(RW, N - r0);
    // Lane l walks row r0 + l's ancestor chain into its bitset (all the
    // warp's walks at once); a checked tree has parents[c] < c, so each ends.
    for (int r = 0; r < nr; ++r)
        for (int w = lane; w < words; w += 32) sh.bits[warp][r][w] = 0u;
    __syncwarp();
    int depth = -1;
    if (lane < nr && ok) {
        uint32_t *bs = sh.bits[warp][lane];
        for (int c = r0 + lane; c >= 0; c = sh.par[c]) {
            bs[c >> 5] |= 1u << (c & 31);
            ++depth;
        }
    }
    __syncwarp();
    if (a.pos && lane < nr)
        a.pos[static_cast<size_t>(b) * N + r0 + lane] = ok ? (a.pos0 ? a.pos0[b] : 0) + depth : -1;
    for (int r = 0; r < nr; ++r) {
        const uint32_t *bs = sh.bits[warp][r];
        const size_t rb = (static_cast<size_t>(b) * N + r0 + r) * N;
        if (a.mask) {
            uint8_t *row = a.mask + rb;
            if (N % 16 == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
                for (int j = lane * 16; j < N; j += 32 * 16) {
                    const uint32_t w16 = bs[j >> 5] >> (j & 31);
                    *reinterpret_cast<uint4 *>(row + j) =
                        make_uint4(bits_to_bytes(w16), bits_to_bytes(w16 >> 4),
                                   bits_to_bytes(w16 >> 8), bits_to_bytes(w16 >> 12));
                }
            } else {
                for (int j = lane; j < N; j += 32)
                    row[j] = static_cast<uint8_t>((bs[j >> 5] >> (j & 31)) & 1u);
            }
        }
        if (a.bias) {
            float *row = a.bias + rb;
            auto val = [&](int j) { return (bs[j >> 5] >> (j & 31)) & 1u ? 0.0f : kNegInf; };
            if (N % 4 == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
                for (int j = lane * 4; j < N; j += 32 * 4)
                    *reinterpret_cast<float4 *>(row + j) =
                        make_float4(val(j), val(j + 1), val(j + 2), val(j + 3));
            } else {
                for (int j = lane; j < N; j += 32) row[j] = val(j);
            }
        }
    }
}

bool tree_mask_smem_ok() {
    constexpr int kMaxDev = 64;
    static int done[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    if (__atomic_load_n(&done[dev], __ATOMIC_RELAXED)) return true;
    if (cudaFuncSetAttribute(tree_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(TreeMaskShared))) != cudaSuccess)
        return false;
    __atomic_store_n(&done[dev], 1, __ATOMIC_RELAXED);
    return true;
}

}  // namespace

int launch_tree_mask(const TreeMaskArgs &a, cudaStream_t st) {
    if (!tree_mask_smem_ok()) return SPEC_ERR_CUDA;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SPEC_ERR_CUDA;
    // Rows per warp: 32 when there are rows enough for two CTAs per SM at
    // that size, fewer (a power of two) for small batches, so that the
    // writes spread over more warps.
    TreeMaskArgs k = a;
    const long long rows = static_cast<long long>(a.B) * a.N;
    k.rows_per_warp = 32;
    while (k.rows_per_warp > 1 && rows < 2LL * sms * kWarps * k.rows_per_warp) k.rows_per_warp /= 2;
    const int cta_rows = kWarps * k.rows_per_warp;
    const long long grid = static_cast<long long>(a.B) * ((a.N + cta_rows - 1) / cta_rows);
    tree_mask_kernel<<<static_cast<unsigned>(grid), kThreads, sizeof(TreeMaskShared), st>>>(k);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
