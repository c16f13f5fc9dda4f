// Retrieval for the RAG draft's compressed context.
//
// "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
// Decoding", section 3.1 (RAG settings): the long context is cut into
// 512-token chunks, each embedded; chunks are ranked by the cosine similarity
// of their embedding with the query embedding, chunks below 0.3 are dropped,
// and the retrieved context stays within at least 4096 tokens and 1/24 of
// the input.  Reading taken here: budget = max(min_tokens, n / ratio); chunks
// are visited in descending score (ties: lower index), the visit stops at the
// first chunk below the threshold, a chunk is kept if its tokens fit what is
// left of the budget, and the kept chunk ids are written in document order.
//
// Scores: each warp streams whole chunk rows with 16-byte loads, all in
// flight before any arithmetic; fp32 sums.
// Selection: one CTA per sequence sorts (score, index) keys in shared memory
// (bitonic), walks the budget, and compacts the kept ids in index order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "retrieval.cuh"

namespace rapid {

namespace {

constexpr int kScoreWarps = 8;   // warps per block of the scores kernel
constexpr int kSelectMaxThreads = 1024;

// Eight elements as four float pairs from kVec16 16-byte words.
__device__ __forceinline__ void to_pairs(const uint4 (&w)[1], float2 (&v)[4], const __nv_bfloat16*) {
    const uint32_t x[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = make_float2(__uint_as_float(x[i] << 16), __uint_as_float(x[i] & 0xffff0000u));
}
__device__ __forceinline__ void to_pairs(const uint4 (&w)[2], float2 (&v)[4], const float*) {
    v[0] = make_float2(__uint_as_float(w[0].x), __uint_as_float(w[0].y));
    v[1] = make_float2(__uint_as_float(w[0].z), __uint_as_float(w[0].w));
    v[2] = make_float2(__uint_as_float(w[1].x), __uint_as_float(w[1].y));
    v[3] = make_float2(__uint_as_float(w[1].z), __uint_as_float(w[1].w));
}

template <typename T>
struct Vec {
    static constexpr int kWords = sizeof(T) == 2 ? 1 : 2;   // 16-byte words per 8 elements
};

// Cosine of each chunk row with its sequence's query.  A warp takes R
// consecutive rows; lane l holds the 8-element pieces at l*8 + u*256.  With
// P > 0 (D <= 256 P) every piece of all R rows is loaded (streaming, evict
// first) before any arithmetic, so a warp keeps R * D elements in flight;
// the query is read once per warp through the read-only path (it stays in
// L1 / L2: one row per sequence).  P == 0 handles longer rows in passes of
// four pieces, one row per warp.  Sums are fp32 pairs (f32x2 FMA).
template <typename T, int P, int R>
__global__ void __launch_bounds__(32 * kScoreWarps, sizeof(T) == 2 ? 4 : 3)
retrieval_scores_kernel(const T* __restrict__ query, const T* __restrict__ chunks, int N, int D,
                        int64_t rows, float* __restrict__ scores) {
    constexpr int W = Vec<T>::kWords;
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = ((int64_t)blockIdx.x * kScoreWarps + warp) * R;
    if (row0 >= rows) return;
    if constexpr (P > 0) {
        uint4 cw[R][P][W];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int u = 0; u < P; ++u) {
                const int k0 = lane * 8 + u * 256;
                if (row0 + j < rows && k0 < D) {
                    const uint4* p = reinterpret_cast<const uint4*>(chunks + (row0 + j) * D + k0);
#pragma unroll
                    for (int v = 0; v < W; ++v) cw[j][u][v] = __ldcs(p + v);
                }
            }
        int64_t qb = -1;
        uint4 qw[P][W];
        float qq = 0.f;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int64_t row = row0 + j;
            if (row >= rows) break;
            const int64_t b = row / N;
            if (b != qb) {
                float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < P; ++u) {
                    const int k0 = lane * 8 + u * 256;
                    if (k0 < D) {
                        const uint4* p = reinterpret_cast<const uint4*>(query + b * D + k0);
#pragma unroll
                        for (int v = 0; v < W; ++v) qw[u][v] = __ldg(p + v);
                        float2 qv[4];
                        to_pairs(qw[u], qv, query);
#pragma unroll
                        for (int i = 0; i < 4; ++i) q2 = fma2(qv[i], qv[i], q2);
                    }
                }
                qq = warp_sum(q2.x + q2.y);
                qb = b;
            }
            float2 qc2 = make_float2(0.f, 0.f), cc2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < P; ++u) {
                if (lane * 8 + u * 256 < D) {
                    float2 qv[4], cv[4];
                    to_pairs(qw[u], qv, query);
                    to_pairs(cw[j][u], cv, query);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qc2 = fma2(qv[i], cv[i], qc2);
                        cc2 = fma2(cv[i], cv[i], cc2);
                    }
                }
            }
            const float qc = warp_sum(qc2.x + qc2.y);
            const float cc = warp_sum(cc2.x + cc2.y);
            if (lane == 0) scores[row] = (qq > 0.f && cc > 0.f) ? qc / (sqrtf(qq) * sqrtf(cc)) : 0.f;
        }
    } else {
        const int64_t row = row0;
        const T* c = chunks + row * D;
        const T* q = query + (row / N) * D;
        float2 q2 = make_float2(0.f, 0.f), qc2 = q2, cc2 = q2;
        for (int k0 = lane * 8; k0 < D; k0 += 4 * 256) {
            uint4 cw[4][W], qw[4][W];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (k0 + u * 256 < D) {
#pragma unroll
                    for (int v = 0; v < W; ++v) {
                        cw[u][v] = __ldcs(reinterpret_cast<const uint4*>(c + k0 + u * 256) + v);
                        qw[u][v] = __ldg(reinterpret_cast<const uint4*>(q + k0 + u * 256) + v);
                    }
                }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (k0 + u * 256 < D) {
                    float2 qv[4], cv[4];
                    to_pairs(qw[u], qv, query);
                    to_pairs(cw[u], cv, query);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        q2 = fma2(qv[i], qv[i], q2);
                        qc2 = fma2(qv[i], cv[i], qc2);
                        cc2 = fma2(cv[i], cv[i], cc2);
                    }
                }
        }
        const float qq = warp_sum(q2.x + q2.y);
        const float qc = warp_sum(qc2.x + qc2.y);
        const float cc = warp_sum(cc2.x + cc2.y);
        if (lane == 0) scores[row] = (qq > 0.f && cc > 0.f) ? qc / (sqrtf(qq) * sqrtf(cc)) : 0.f;
    }
}

// Key whose unsigned order is (score descending, index ascending) when
// sorted in descending order.
__device__ __forceinline__ uint64_t make_key(float s, int idx) {
    if (s == 0.f) s = 0.f;   // -0 and +0 compare equal
    uint32_t u = __float_as_uint(s);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)u << 32) | (uint64_t)(0xffffffffu - (uint32_t)idx);
}
__device__ __forceinline__ float key_score(uint64_t k) {
    uint32_t u = (uint32_t)(k >> 32);
    u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
    return __uint_as_float(u);
}
__device__ __forceinline__ int key_index(uint64_t k) {
    return (int)(0xffffffffu - (uint32_t)k);
}

__global__ void __launch_bounds__(kSelectMaxThreads)
retrieval_select_kernel(const float* __restrict__ scores, const int32_t* __restrict__ context_tokens,
                        int N, int chunk, float threshold, int min_tokens, int ratio,
                        int32_t* __restrict__ selected, int32_t* __restrict__ n_selected,
                        int32_t* __restrict__ tokens_selected, unsigned int* err) {
    extern __shared__ uint64_t keys[];   // [P2] sort keys, then keep flags [N] after them
    __shared__ int s_pos[kSelectMaxThreads];
    __shared__ int s_cnt, s_tok, s_bad;
    griddep_wait();
    const int b = blockIdx.x;
    const int t = threadIdx.x;
    const int nt = blockDim.x;
    const int64_t n = context_tokens[b];
    const int64_t nc64 = n > 0 ? (n + chunk - 1) / chunk : 0;
    const bool bad = n < 0 || nc64 > N;
    const int nc = bad ? 0 : (int)nc64;
    int P2 = 1;
    while (P2 < nc) P2 <<= 1;
    int P2n = 1;
    while (P2n < N) P2n <<= 1;
    uint8_t* keep = reinterpret_cast<uint8_t*>(keys + P2n);
    const float* s = scores + (int64_t)b * N;
    for (int i = t; i < nc; i += nt) keep[i] = 0;
    for (int i = t; i < P2; i += nt) keys[i] = i < nc ? make_key(s[i], i) : 0ull;
    __syncthreads();
    // bitonic sort, descending
    for (int size = 2; size <= P2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = t; i < P2 / 2; i += nt) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint64_t a = keys[lo], c = keys[hi];
                if ((a < c) == desc) {
                    keys[lo] = c;
                    keys[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    // the budget walk (one thread)
    if (t == 0) {
        const int64_t budget = n / ratio > (int64_t)min_tokens ? n / ratio : (int64_t)min_tokens;
        int64_t left = budget, used = 0;
        int cnt = 0;
        const int64_t last_len = nc > 0 ? n - (int64_t)(nc - 1) * chunk : 0;   // tokens of the last chunk
        bool last_seen = false;
        for (int r = 0; r < nc; ++r) {
            const uint64_t k = keys[r];
            if (!(key_score(k) >= threshold)) break;
            const int idx = key_index(k);
            const int64_t len = idx == nc - 1 ? last_len : chunk;
            if (idx == nc - 1) last_seen = true;
            if (len <= left) {
                keep[idx] = 1;
                ++cnt;
                left -= len;
                used += len;
            }
            if (left < chunk) {
                // no whole chunk fits any more; a short last chunk is kept if the
                // walk would reach it (its score is at or above the threshold)
                if (!last_seen && last_len < chunk && last_len <= left && s[nc - 1] >= threshold) {
                    keep[nc - 1] = 1;
                    ++cnt;
                    used += last_len;
                }
                break;
            }
        }
        s_cnt = cnt;
        s_tok = (int)used;
        s_bad = bad ? 1 : 0;
    }
    __syncthreads();
    const int cnt = s_cnt;
    // compaction in index order: each thread counts a contiguous run of flags
    const int per = (nc + nt - 1) / nt;
    const int a0 = min(nc, t * per), a1 = min(nc, a0 + per);
    int mine = 0;
    for (int i = a0; i < a1; ++i) mine += keep[i];
    s_pos[t] = mine;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {   // inclusive scan (Hillis-Steele)
        const int v = t >= off ? s_pos[t - off] : 0;
        __syncthreads();
        s_pos[t] += v;
        __syncthreads();
    }
    int w = s_pos[t] - mine;
    int32_t* out = selected + (int64_t)b * N;
    for (int i = a0; i < a1; ++i)
        if (keep[i]) out[w++] = i;
    for (int i = cnt + t; i < N; i += nt) out[i] = -1;
    if (t == 0) {
        n_selected[b] = cnt;
        tokens_selected[b] = s_tok;
        if (s_bad && err) atomicOr(err, kErrBadInput);
    }
}

template <typename T, int P, int R>
cudaError_t launch_scores_typed(const void* query, const void* chunks, int B, int N, int D,
                                float* scores, cudaStream_t st) {
    const int64_t rows = (int64_t)B * N;
    const int64_t per_block = (int64_t)kScoreWarps * R;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + per_block - 1) / per_block), 1, 1);
    cfg.blockDim = dim3(32 * kScoreWarps, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, retrieval_scores_kernel<T, P, R>, static_cast<const T*>(query),
                              static_cast<const T*>(chunks), N, D, rows, scores);
}

template <typename T>
cudaError_t launch_scores_dispatch(const void* query, const void* chunks, int B, int N, int D,
                                   float* scores, cudaStream_t st) {
    // two rows per warp for bf16 (the same registers as one fp32 row)
    constexpr int R = sizeof(T) == 2 ? 2 : 1;
    switch ((D + 255) / 256) {   // pieces of 8 elements per lane
        case 1: return launch_scores_typed<T, 1, R>(query, chunks, B, N, D, scores, st);
        case 2: return launch_scores_typed<T, 2, R>(query, chunks, B, N, D, scores, st);
        case 3: return launch_scores_typed<T, 3, R>(query, chunks, B, N, D, scores, st);
        case 4: return launch_scores_typed<T, 4, R>(query, chunks, B, N, D, scores, st);
        default: return launch_scores_typed<T, 0, 1>(query, chunks, B, N, D, scores, st);
    }
}

}  // namespace

cudaError_t launch_retrieval_scores(const void* query, const void* chunks, int dtype, int B, int N,
                                    int D, float* scores, cudaStream_t st) {
    return dtype == 1 ? launch_scores_dispatch<__nv_bfloat16>(query, chunks, B, N, D, scores, st)
                      : launch_scores_dispatch<float>(query, chunks, B, N, D, scores, st);
}

cudaError_t launch_retrieval_select(const float* scores, const int32_t* context_tokens, int B, int N,
                                    int chunk, float threshold, int min_tokens, int ratio,
                                    int32_t* selected, int32_t* n_selected,
                                    int32_t* tokens_selected, unsigned int* err, cudaStream_t st) {
    int P2 = 1;
    while (P2 < N) P2 <<= 1;
    const size_t smem = (size_t)P2 * sizeof(uint64_t) + (size_t)((N + 15) / 16 * 16);
    cudaError_t e = cudaFuncSetAttribute(retrieval_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    // one thread per compare-exchange pair of the widest sort, at least a warp
    const int threads = P2 / 2 < 32 ? 32 : (P2 / 2 > kSelectMaxThreads ? kSelectMaxThreads : P2 / 2);
    cfg.gridDim = dim3(B, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, retrieval_select_kernel, scores, context_tokens, N, chunk,
                              threshold, min_tokens, ratio, selected, n_selected, tokens_selected,
                              err);
}

}  // namespace rapid
