// Acceptance kernels: parameter block and launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rapid {

constexpr int kAcceptThreads = 256;
constexpr int kAcceptMaxNq = 64;

struct AcceptParams {
    const float* z;              // [B, n_q, V] target logits
    const float* q;              // [B, n_q, V] draft probabilities
    const int32_t* tokens;       // [B, n_q]
    const int32_t* parent;       // [B, n_q] or nullptr (chain)
    int32_t* ws_accept;          // [B, n_q] ratio-test outcome of node i
    int32_t* ws_sample;          // [B, n_q] candidate next token drawn from row j
    float* diag;                 // [B, n_q, 5] or nullptr
    int32_t* n_accepted;         // [B]
    int32_t* next_token;         // [B]
    int32_t* path;               // [B, n_q] or nullptr
    unsigned int* err;           // sticky device error word
    int B, n_q, V;
    int chunk;                   // vocabulary entries per CTA (multiple of 4)
    int bulk;                    // 1: rows 16-byte aligned, use bulk copies
    int clamp;                   // tail rule on/off
    float invT, eta;
    uint32_t seed_lo, seed_hi;
};

struct AcceptShape {
    int vocab;     // V
    int cluster;   // CTAs per row (thread-block cluster size)
    int chunk;     // entries per CTA
    int F;         // float4 groups per thread
};

// Default split of a row of V entries over a cluster (1..16 CTAs).
AcceptShape accept_shape(int V, int preferred_cluster);
// Shrink the cluster until the device can schedule it.
cudaError_t accept_check_cluster(AcceptShape* sh);
// Row kernel + selection kernel on stream st.
cudaError_t launch_accept(const AcceptParams& p, const AcceptShape& sh, cudaStream_t st);

}  // namespace rapid
