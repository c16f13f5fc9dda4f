// rapid_accept_noalloc: the acceptance step with its scratch memory in a
// statically allocated device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// acceptance step: a host framework that owns all device memory and hands its
// plug-ins no allocator, or a latency-critical decode loop that must never
// call cudaMalloc (which may synchronise the device).  For them this entry
// point takes only inputs and outputs.  Its scratch (per node: the ratio-test
// outcome and the row's softmax statistics, 20 bytes; 80 KB for 4096 nodes)
// lives in the array
// below, which every GPU that loads librapid.so holds until the process
// exits.  The verification step of the pages has no counterpart of this; it
// is a packaging variant of rapid_accept.
#include <cuda_runtime.h>

#include "rapid.h"

namespace rapid {
namespace {

constexpr size_t align256(size_t n) { return (n + 255) / 256 * 256; }
// The layout rapid_accept_workspace_size describes.
constexpr size_t kNodes = (size_t)RAPID_NOALLOC_MAX_NODES;
constexpr size_t kScratchBytes = align256(kNodes * sizeof(int32_t)) +
                                 align256(kNodes * 4 * sizeof(float));

// Shared by every call on a device; see the concurrency note in rapid.h.
static __device__ __align__(256) unsigned char g_accept_scratch[kScratchBytes];

// Device address of g_accept_scratch on the current device.  In host code the
// name g_accept_scratch is only a host-side stand-in, never a device address.
// It is looked up on every call (cudaGetSymbolAddress allocates nothing and
// costs well under a microsecond once the module is loaded), so a device
// reset or a re-created context never leaves a stale cached address.
void* scratch_address() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_accept_scratch) != cudaSuccess || ptr == nullptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return ptr;
}

}  // namespace
}  // namespace rapid

extern "C" rapid_status rapid_accept_noalloc(const float* z_target, const float* q_draft,
                                             const int32_t* draft_tokens, const int32_t* parent,
                                             int B, int n_q, int V, float T, float eta,
                                             uint64_t philox_seed, uint32_t flags,
                                             int32_t* n_accepted, int32_t* next_token,
                                             int32_t* path, float* diag, void* stream) {
    if (B < 1 || n_q < 1 || n_q > RAPID_MAX_NQ) return RAPID_EINVAL;
    if ((int64_t)B * n_q > RAPID_NOALLOC_MAX_NODES) return RAPID_EUNSUPPORTED;
    void* scratch = rapid::scratch_address();
    if (!scratch) return RAPID_ECUDA;
    // Nothing in the scratch needs to start at zero: every entry that the
    // selection kernel reads is written earlier in the same call.
    return rapid_accept(z_target, q_draft, draft_tokens, parent, B, n_q, V, T, eta, philox_seed,
                        flags, n_accepted, next_token, path, diag, scratch,
                        rapid::kScratchBytes, stream);
}
