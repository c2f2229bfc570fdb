// noalloc.cu -- spec_verify_sample_noalloc: spec_verify_sample for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they verify: a
// serving engine that plans every device buffer up front and forbids
// allocation on its decode path, a plugin whose host framework owns all
// device memory and gives it no allocator, or a latency-critical loop that
// cannot afford cudaMalloc's implicit synchronisation.  Such a caller
// cannot hand spec_verify_sample a workspace of its own.  This entry point
// uses a fixed scratch array that lives in the library's own device image
// instead: every GPU that loads the library holds kNoAllocScratchBytes of
// it until the process exits, and this file allocates nothing.
//
// Sharing and ordering: all calls on one device share the one array, and it
// keeps the previous call's contents.  Each call first zero-fills the part
// it will use (cudaMemsetAsync on the caller's stream, not an allocation),
// so its counters start at zero.  Two calls whose work overlaps on the GPU
// (different streams without ordering between them) race on the array and
// give wrong results: order them.
//
// Set-up: the first call on a device, with that device current, looks up
// the array's device address (cudaGetSymbolAddress) and caches it for that
// device.  Make that first call before any stream capture begins.  The
// cached address belongs to the device's primary context, which the CUDA
// runtime keeps for the life of the process: a caller that destroys it
// (cudaDeviceReset) must not use this entry point on that device again in
// the same process, since the cache would still hold the old address.

#include <mutex>

#include "common.cuh"

#define SPEC_EXPORT extern "C" __attribute__((visibility("default")))

namespace specv {
// Workspace bytes a chain call needs (api.cu), with or without top-k.
size_t chain_workspace_bytes(int B, int k, int V, bool topk);
}  // namespace specv

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol,
// not a device address: the address is obtained with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per
// device); nullptr if the lookup failed.
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

SPEC_EXPORT int spec_verify_sample_noalloc(const void *target_logits, const void *draft_logits,
                                           const int32_t *draft_tokens, const float *uniforms,
                                           int B, int k, int V, float temperature, float top_p,
                                           int mode, int dtype, int32_t *out_tokens,
                                           int32_t *out_num_accepted, spec_stream_t stream) {
    size_t need = 0;
    const int rc = spec_verify_workspace_size(B, k, V, &need);
    if (rc != SPEC_OK) return rc;
    // B = 0: spec_verify_sample checks the mode, dtype and sizes, enqueues
    // nothing and touches no pointer.
    if (B == 0)
        return spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, B, k, V,
                                  temperature, top_p, mode, dtype, out_tokens, out_num_accepted,
                                  nullptr, 0, stream);
    need = specv::chain_workspace_bytes(B, k, V, false);  // no top-k: not the summaries
    if (need > kNoAllocScratchBytes) return SPEC_ERR_WORKSPACE;  // batch too large for the scratch
    void *scratch = scratch_on_current_device();
    if (!scratch) return SPEC_ERR_CUDA;
    // Validate every other argument without enqueueing anything:
    // spec_verify_sample checks the workspace size last, so with a size of
    // 0 it answers SPEC_ERR_WORKSPACE exactly when all else is valid.
    const int pre = spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, B, k,
                                       V, temperature, top_p, mode, dtype, out_tokens,
                                       out_num_accepted, scratch, 0, stream);
    if (pre != SPEC_ERR_WORKSPACE) return pre;
    if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, B, k, V,
                              temperature, top_p, mode, dtype, out_tokens, out_num_accepted,
                              scratch, kNoAllocScratchBytes, stream);
}
