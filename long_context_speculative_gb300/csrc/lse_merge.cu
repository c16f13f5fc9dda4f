// Log-sum-exp merge of partial attention results over disjoint key sets.
//
// "LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", section 2.3 (Hybrid Tree Attention): the
// history part and the speculative part are computed separately and combined
// through their log-sum-exp.  The same combine takes any number of parts:
// with L_p the natural-log log-sum-exp of part p's scores and O_p its
// normalised output, L = ln sum_p e^{L_p} and O = sum_p e^{L_p - L} O_p.  A
// part with L_p = -inf saw no key and has weight 0; a row left with no part
// gets O = 0 and L = -inf.  rapid_verify_attn merges its own splits
// internally; this kernel merges results that were computed separately
// (other shards of the key range, possibly on other devices).
#include <cuda_bf16.h>

#include "common.cuh"
#include "lse_merge.cuh"

namespace rapid {

namespace {

constexpr int kMergeWarps = 8;   // rows per 256-thread block
constexpr int kMergeBatch = 8;   // parts loaded at once per lane

// V consecutive elements of a row as floats (V = 2 or 4).
template <int V>
RAPID_DEVICE void load_vec(const float* p, float (&x)[V]) {
    if constexpr (V == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x; x[1] = v.y;
    }
}
template <int V>
RAPID_DEVICE void load_vec(const __nv_bfloat16* p, float (&x)[V]) {
    if constexpr (V == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
        x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(v << 16); x[1] = __uint_as_float(v & 0xffff0000u);
    }
}
template <int V>
RAPID_DEVICE void store_vec(float* p, const float (&x)[V]) {
    if constexpr (V == 4) *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    else *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
}
template <int V>
RAPID_DEVICE void store_vec(__nv_bfloat16* p, const float (&x)[V]) {
#pragma unroll
    for (int c = 0; c < V; ++c) p[c] = from_float<__nv_bfloat16>(x[c]);
}

// One warp per row; lane l holds columns l V .. l V + V - 1 (V = D / 32).
// The row's largest part LSE first (lanes split the parts), then the parts
// in batches whose loads are all in flight before the sums.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kMergeWarps)
lse_merge_kernel(const T* __restrict__ O_parts, const float* __restrict__ LSE_parts, int n_parts,
                 int64_t rows, T* __restrict__ O, float* __restrict__ LSE) {
    constexpr int V = D / 32;
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    float m = -INFINITY;
    for (int p = lane; p < n_parts; p += 32) m = fmaxf(m, LSE_parts[(int64_t)p * rows + row]);
    m = warp_max(m);
    float acc[V];
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] = 0.f;
    float s = 0.f;
    if (m != -INFINITY) {
        for (int p0 = 0; p0 < n_parts; p0 += kMergeBatch) {
            float lp[kMergeBatch], x[kMergeBatch][V];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const int p = p0 + u;
                lp[u] = p < n_parts ? LSE_parts[(int64_t)p * rows + row] : -INFINITY;
                if (lp[u] != -INFINITY) {
                    load_vec<V>(O_parts + ((int64_t)p * rows + row) * D + lane * V, x[u]);
                } else {
#pragma unroll
                    for (int c = 0; c < V; ++c) x[u][c] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const float w = lp[u] != -INFINITY ? expf(lp[u] - m) : 0.f;
                s += w;
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = fmaf(w, x[u][c], acc[c]);
            }
        }
    }
    const float inv = s > 0.f ? 1.f / s : 0.f;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] *= inv;
    store_vec<V>(O + row * D + lane * V, acc);
    if (lane == 0) LSE[row] = s > 0.f ? m + logf(s) : -INFINITY;
}

template <typename T, int D>
cudaError_t launch_typed(const void* O_parts, const float* LSE_parts, int n_parts, int64_t rows,
                         void* O, float* LSE, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kMergeWarps - 1) / kMergeWarps), 1, 1);
    cfg.blockDim = dim3(32 * kMergeWarps, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, D>, static_cast<const T*>(O_parts),
                              LSE_parts, n_parts, rows, static_cast<T*>(O), LSE);
}

}  // namespace

cudaError_t launch_lse_merge(const void* O_parts, const float* LSE_parts, bool bf16, int n_parts,
                             int64_t rows, int d, void* O, float* LSE, cudaStream_t st) {
    if (bf16) {
        return d == 64 ? launch_typed<__nv_bfloat16, 64>(O_parts, LSE_parts, n_parts, rows, O, LSE, st)
                       : launch_typed<__nv_bfloat16, 128>(O_parts, LSE_parts, n_parts, rows, O, LSE, st);
    }
    return d == 64 ? launch_typed<float, 64>(O_parts, LSE_parts, n_parts, rows, O, LSE, st)
                   : launch_typed<float, 128>(O_parts, LSE_parts, n_parts, rows, O, LSE, st);
}

}  // namespace rapid
