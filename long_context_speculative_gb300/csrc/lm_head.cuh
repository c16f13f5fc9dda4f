// Target logits of the verify rows from the shared LM head: launcher.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rapid {

// True when the driver's tensor-map encoder is available.
bool lm_head_supported();

// z[r][v] = sum_k hidden[r][k] * W[v][k] for r < rows, v < V; hidden [rows,
// hidden_dim] and W [V, hidden_dim] bf16, z [rows, V] fp32.  rows <= 256 (the
// MMA's N, padded to 16..256), hidden_dim a multiple of 64; hidden, W 16-byte
// aligned.
cudaError_t launch_lm_head(const void* hidden, const void* W, int rows, int hidden_dim, int V,
                           float* z, unsigned int* err, cudaStream_t st);

// The acceptance step on the logits of rapid_lm_head inside the same kernel
// (rows = B * n_q <= kLmFusedMaxRows): every CTA keeps its vocabulary run of
// z and of q in shared memory, and the vocabulary-wide softmax statistics,
// the ratio tests, the path selection and the residual draw run after the
// product, separated by three grid-wide barriers.  z never leaves the chip.
constexpr int kLmFusedMaxRows = 16;

struct LmAcceptParams {
    const float* q;                       // [B * n_q, V] draft probabilities
    const int32_t* tokens;                // [B, n_q]
    const int32_t* parent;                // [B, n_q] or nullptr (chain)
    const int32_t* n_nodes;               // [B] or nullptr
    const unsigned long long* seed_dev;   // device Philox key or nullptr
    int32_t* n_accepted;                  // [B]
    int32_t* next_token;                  // [B]
    int32_t* path;                        // [B, n_q] or nullptr
    float* diag;                          // [B, n_q, 5] or nullptr
    // scratch (the call's workspace)
    unsigned int* bar;                    // grid-barrier arrival count, zeroed before the launch
    float2* part1;                        // [grid, rows] (max, sum) of z / T per CTA
    float2* part2;                        // [grid, rows] (max, sum) of the augmented logits per CTA
    float2* part3;                        // [grid, B] residual and p mass of row e per CTA
    float2* zq_tok;                       // [rows] (z, q) at node i's token in its parent's row
    int B, n_q, clamp;
    int stages;                           // K/V ring stages that fit beside z and q
    int run_max;                          // vocabulary entries per CTA (row pitch of z and q)
    float invT, eta;
    uint32_t seed_lo, seed_hi;
};

// Bytes of the fused call's scratch for `grid` CTAs.
size_t lm_accept_scratch_bytes(int grid, int rows, int B);

// Launches the fused kernel if this shape and device allow it (rows <= 16,
// V % 4 == 0, q 16-byte aligned, every CTA co-resident); otherwise returns
// cudaErrorNotSupported and launches nothing.  The caller fills every field
// of `fa` but the scratch pointers, stages and run_max, which come from
// `scratch` (256-byte aligned; too few bytes: cudaErrorNotSupported).
cudaError_t launch_lm_head_accept(const void* hidden, const void* W, int hidden_dim, int V,
                                  LmAcceptParams fa, void* scratch, size_t scratch_bytes,
                                  unsigned int* err, cudaStream_t st);

}  // namespace rapid
