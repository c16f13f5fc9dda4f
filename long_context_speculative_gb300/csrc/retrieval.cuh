// Retrieval for the RAG draft's compressed context: launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rapid {

constexpr int kRetrievalMaxChunks = 8192;

cudaError_t launch_retrieval_scores(const void* query, const void* chunks, int dtype, int B, int N,
                                    int D, float* scores, cudaStream_t st);
cudaError_t launch_retrieval_select(const float* scores, const int32_t* context_tokens, int B, int N,
                                    int chunk, float threshold, int min_tokens, int ratio,
                                    int32_t* selected, int32_t* n_selected,
                                    int32_t* tokens_selected, unsigned int* err, cudaStream_t st);

}  // namespace rapid
