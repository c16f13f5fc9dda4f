// Verify attention: shared parameter block and kernel entry points.
//
// Hybrid tree attention ("LongSpec: Long-Context Lossless Speculative Decoding
// with Efficient Drafting and Verification", section 2.3): the history rows
// [0, prefix_len) are attended without a mask, split across CTAs (split-KV)
// that each leave an un-normalised partial (acc, m, l) in the workspace; the
// n_q speculative rows are attended under the chain/tree mask inside the merge
// kernel, which then combines all partials by log-sum-exp.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rapid {

struct AttnParams {
    const void* Q;        // [B, Hq, n_q, d]
    const void* K;        // [B, Hkv, cap, d]
    const void* V;        // [B, Hkv, cap, d]
    const int32_t* prefix_len;  // [B]
    const uint8_t* mask;  // [B, n_q, n_q] or nullptr (chain)
    void* O;              // [B, Hq, n_q, d]
    float* LSE;           // [B, Hq, n_q]
    float* part_acc;      // [B*Hkv, nparts, R, d]   un-normalised partial outputs
    float* part_ml;       // [B*Hkv, nparts, R, 2]   (running max m, sum l), log2 domain
    unsigned int* err;    // sticky device error word
    int64_t cap;          // KV rows per head
    int64_t chunk;        // history rows per split (multiple of 128)
    int B, Hq, Hkv, d, n_q, G, R, S;
    int spec_in_partials; // 1: the history kernel already attended the speculative rows
    int nparts;           // partial slots per (b, KV head): S, or 2 S for the tensor-core kernel
    float scale;          // softmax scale (natural units)
    float scale_log2;     // scale * log2(e)
};

// History length of sequence b, clamped so every access stays in the cache.
__device__ __forceinline__ int64_t clamped_prefix(const AttnParams& p, int b) {
    int64_t P = p.prefix_len[b];
    if (P < 0) P = 0;
    if (P > p.cap - p.n_q) P = p.cap - p.n_q;
    return P;
}

// Launchers (return cudaError_t of the launch).
cudaError_t launch_attn_prefix_simt(const AttnParams& p, int dtype, cudaStream_t s);
cudaError_t launch_attn_merge(const AttnParams& p, int dtype, cudaStream_t s);
// tcgen05 + TMA prefix kernel (bf16, d = 128, R <= 128).  Returns
// cudaErrorNotSupported when the shape is outside what it handles.
cudaError_t launch_attn_prefix_tc(const AttnParams& p, cudaStream_t s);
bool attn_prefix_tc_supported(const AttnParams& p, int dtype);

}  // namespace rapid
