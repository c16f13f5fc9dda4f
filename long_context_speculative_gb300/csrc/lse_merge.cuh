// Log-sum-exp merge of separately computed attention parts (rapid_attn_merge).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace rapid {

// O_parts [n_parts, rows, d] (bf16 or fp32), LSE_parts [n_parts, rows] ->
// O [rows, d] (same type), LSE [rows]; d is 64 or 128.
cudaError_t launch_lse_merge(const void* O_parts, const float* LSE_parts, bool bf16, int n_parts,
                             int64_t rows, int d, void* O, float* LSE, cudaStream_t st);

}  // namespace rapid
