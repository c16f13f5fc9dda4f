// Acceptance kernels: parameter block and launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rapid {

constexpr int kAcceptRowThreads = 1024;   // threads of a row-kernel CTA
constexpr int kAcceptSelThreads = 512;    // threads of a selection-kernel CTA
constexpr int kAcceptMaxNq = 64;
constexpr int kAcceptMaxCluster = 16;
constexpr int kAcceptMaxF = 7;            // float4 groups per row-kernel thread
constexpr int kAcceptMaxSlice = 14336;    // entries per CTA (two resident rows of z and q)

struct AcceptParams {
    const float* z;              // [B, n_q, V] target logits
    const float* q;              // [B, n_q, V] draft probabilities
    const int32_t* tokens;       // [B, n_q]
    const int32_t* parent;       // [B, n_q] or nullptr (chain)
    int32_t* ws_accept;          // [B * n_q] ratio-test outcome of node i
    float* ws_stats;             // [B * n_q, 4] (m1, s1), (m2, s2) of row j: softmax = exp(. - m) / s
    float* diag;                 // [B, n_q, 5] or nullptr
    int32_t* n_accepted;         // [B]
    int32_t* next_token;         // [B]
    int32_t* path;               // [B, n_q] or nullptr
    unsigned int* err;           // sticky device error word
    int B, n_q, V;
    int rows;                    // B * n_q
    int chunk;                   // vocabulary entries per CTA (multiple of 4)
    int groups;                  // float4 groups per shared-memory row array (multiple of 32)
    int C;                       // CTAs per cluster (one vocabulary slice each)
    int nclusters;               // persistent clusters; cluster c takes rows c, c + nclusters, ...
    int nbuf;                    // rows of (z, q) resident per CTA (>= 2)
    int bulk;                    // 1: rows 16-byte aligned, use bulk copies
    int clamp;                   // tail rule on/off
    float invT, eta;
    uint32_t seed_lo, seed_hi;
    // non-null: the key is read from here when the kernels run (seed_lo and
    // seed_hi unused), so a call captured in a graph sees the current value
    const unsigned long long* seed_dev;
    // non-null: sequence b has n_nodes[b] nodes (clamped to [1, n_q]); the
    // nodes past it take no part in the selection
    const int32_t* n_nodes;
};

struct AcceptShape {
    int vocab;          // V
    int cluster;        // CTAs per cluster
    int chunk;          // entries per CTA
    int groups;         // float4 groups per shared-memory row array
    int F;              // float4 groups per thread
    int nbuf;           // resident rows per CTA
    int max_clusters;   // co-resident clusters of this shape on the current device
};

// Choose the cluster size for `rows` rows of V entries on the current
// device: among the slice counts whose slice fits the compiled kernels, the
// one with the least vocabulary per cluster to stream (rows per cluster x
// slice length).  Fails if no shape can be co-scheduled.
cudaError_t accept_plan(int V, int rows, AcceptShape* sh);
// Row kernel + selection kernel on stream st.
cudaError_t launch_accept(const AcceptParams& p, const AcceptShape& sh, cudaStream_t st);

}  // namespace rapid
