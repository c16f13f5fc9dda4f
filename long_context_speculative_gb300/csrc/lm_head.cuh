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

}  // namespace rapid
