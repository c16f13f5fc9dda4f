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
    // Partials: un-normalised outputs (part_acc, d floats per row) and their
    // (running max m, sum l) in the log2 domain (part_ml, 2 floats per row).
    // CUDA-core kernel: [B*Hkv, nparts, R, .] (every sequence has nparts
    // splits).  Tensor-core kernel: [Hkv, nparts, R, .] by the launch's
    // (sequence, split) slot, nparts = the slots per KV head; sequence b's
    // S_b splits sit at slots part_first[b*Hkv+g] .. + part_nsplit[b*Hkv+g] - 1.
    float* part_acc;
    float* part_ml;
    int* part_nsplit;     // [B*Hkv] splits written per (b, KV head) by the tensor-core kernel
    int* part_first;      // [B*Hkv] first slot of those splits
    unsigned int* err;    // sticky device error word
    int64_t cap;          // KV rows per head
    int64_t chunk;        // history rows per split (multiple of 128)
    int B, Hq, Hkv, d, n_q, G, R, S;
    int spec_in_partials; // 1: the history kernel already attended the speculative rows
    int nparts;           // partial slots per (b, KV head)
    int balanced;         // 1: splits follow split_of() with pairs = S (tensor-core kernel)
    float scale;          // softmax scale (natural units)
    float scale_log2;     // scale * log2(e)
};

// History length of sequence b, clamped so every access stays in the cache.
// (The merge kernel flags an out-of-range value in the device error word.)
__device__ __forceinline__ int64_t clamped_prefix(const AttnParams& p, int b) {
    int64_t P = p.prefix_len[b];
    if (P < 0) P = 0;
    if (P > p.cap - p.n_q) P = p.cap - p.n_q;
    return P;
}

// Balanced split plan of the tensor-core history kernel, computed the same
// way by every CTA and by the merge kernel from the device-side prefix
// lengths: every split gets about the same number of 64-key tiles, so short
// and long sequences of a ragged batch finish together.  `pairs` is the
// number of (sequence, split) slots the launch provides per KV head.
struct SplitOf {
    int b;        // sequence, or -1 when the slot has no work
    int s;        // split of that sequence
    int S_b;      // splits of that sequence
    int tiles;    // 64-key history tiles of that sequence
};

__device__ __forceinline__ int seq_tiles(const AttnParams& p, int b) {
    return (int)((clamped_prefix(p, b) + 63) >> 6);
}

__device__ __forceinline__ int seq_splits(int tiles, int budget) {
    const int S = (tiles + budget - 1) / budget;
    return S < 1 ? 1 : S;
}

// Smallest tile budget whose splits fit in `pairs` slots (binary search;
// budget = the longest sequence always fits because pairs >= B).
__device__ __forceinline__ int split_budget(const AttnParams& p, int pairs) {
    if (p.B == 1) {
        const int t = seq_tiles(p, 0);
        const int budget = (t + pairs - 1) / pairs;
        return budget < 1 ? 1 : budget;
    }
    int total = 0, longest = 1;
    for (int b = 0; b < p.B; ++b) {
        const int t = seq_tiles(p, b);
        total += t;
        longest = t > longest ? t : longest;
    }
    int lo = (total + pairs - 1) / pairs;
    if (lo < 1) lo = 1;
    int hi = longest > lo ? longest : lo;
    while (lo < hi) {
        const int mid = lo + (hi - lo) / 2;
        int used = 0;
        for (int b = 0; b < p.B; ++b) used += seq_splits(seq_tiles(p, b), mid);
        if (used <= pairs) hi = mid; else lo = mid + 1;
    }
    return lo;
}

__device__ __forceinline__ SplitOf split_of(const AttnParams& p, int pairs, int c) {
    const int budget = split_budget(p, pairs);
    int first = 0;
    for (int b = 0; b < p.B; ++b) {
        const int tiles = seq_tiles(p, b);
        const int S_b = seq_splits(tiles, budget);
        if (c < first + S_b) return SplitOf{b, c - first, S_b, tiles};
        first += S_b;
    }
    return SplitOf{-1, 0, 0, 0};
}

// Row blocks of the tensor-core kernel for a group of R rows: one CTA per
// (split, block) covers up to 128 rows, or 256 (two row blocks that share
// every K/V tile) when the group has more than 128.
__host__ __device__ __forceinline__ int tc_row_blocks(int R) {
    const int per_cta = R <= 128 ? 128 : 256;
    return (R + per_cta - 1) / per_cta;
}

// Launchers (return cudaError_t of the launch).
cudaError_t launch_attn_prefix_simt(const AttnParams& p, int dtype, cudaStream_t s);
cudaError_t launch_attn_merge(const AttnParams& p, int dtype, cudaStream_t s);
// tcgen05 + TMA prefix kernel (bf16 caches, d = 64 or 128, up to 512 group
// rows R = G * n_q, run as blocks of 128 rows, or of 256 above 128 rows).  attn_prefix_tc_supported() says
// whether a shape is one it handles.
cudaError_t launch_attn_prefix_tc(const AttnParams& p, cudaStream_t s);
bool attn_prefix_tc_supported(const AttnParams& p, int dtype);

}  // namespace rapid
