// KV commit after a verify step: parameter block and launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rapid {

constexpr int kCommitMaxLayers = 128;

struct CommitParams {
    void* K[kCommitMaxLayers];     // per layer: [B, Hkv, cap, d] cache
    void* V[kCommitMaxLayers];
    const int32_t* prefix_len;     // [B] history length before the step (the root's row)
    const int32_t* path;           // [B, n_q] accepted node ids, root-to-leaf
    const int32_t* n_acc;          // [B]
    int32_t* prefix_out;           // [B] or nullptr: prefix_len + 1 + n_acc
    unsigned int* err;             // sticky device error word
    int64_t cap;
    int layers, B, Hkv, n_q;
    int row_bytes;                 // d * element size (a multiple of 16)
};

cudaError_t launch_kv_commit(const CommitParams& p, cudaStream_t st);
cudaError_t launch_kv_advance(int32_t* prefix_len, const int32_t* n_acc, int B, int n_q,
                              int64_t cap, unsigned int* err, cudaStream_t st);

}  // namespace rapid
