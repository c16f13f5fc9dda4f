// KV commit after a verify step.
//
// In the verify pass the n_q speculative tokens of a step sit after the
// history in every layer's cache, node i at row P + i with node 0 the root
// ("LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", section 2.3).  Once acceptance has chosen a
// root-to-leaf path, its rows -- already computed by the verify pass -- join
// the history right after the root, in path order: row P + 1 + k takes the
// row of node path[k].  The other speculative rows are dropped by not
// counting them (the history grows by 1 + n_accepted) and are overwritten by
// the next step.  A chain's path is 1, 2, ..., so it is already in place.
//
// One CTA per (sequence, KV head, layer) stages the accepted K and V rows in
// shared memory before writing any of them, so a destination that is also a
// later source (path 2, 3, ... shifts every row by one) is read first.
#include "common.cuh"
#include "kv_commit.cuh"

namespace rapid {

namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(const CommitParams p) {
    extern __shared__ uint4 staged[];   // [2, n_q - 1, row_bytes / 16]: K rows, then V rows
    __shared__ int s_src[64];
    __shared__ int s_flags;             // bit 0: invalid input, bit 1: some row moves
    griddep_wait();
    const int t = threadIdx.x;
    const int b = blockIdx.x / p.Hkv;
    const int h = blockIdx.x - b * p.Hkv;
    const int layer = blockIdx.y;
    const int n = p.n_acc[b];
    const int64_t P = p.prefix_len[b];
    if (t == 0) {
        const bool ok = n >= 0 && n <= p.n_q - 1 && P >= 0 && P + p.n_q <= p.cap;
        s_flags = ok ? 0 : 1;
    }
    __syncthreads();
    if (!(s_flags & 1) && t < n) {
        const int src = p.path[(int64_t)b * p.n_q + t];
        const int prev = t > 0 ? p.path[(int64_t)b * p.n_q + t - 1] : 0;
        int f = 0;
        if (src < t + 1 || src > p.n_q - 1 || src <= prev) f |= 1;   // not a valid increasing path
        if (src != t + 1) f |= 2;
        s_src[t] = src;
        if (f) atomicOr(&s_flags, f);
    }
    __syncthreads();
    const int flags = s_flags;
    if (flags & 1) {
        if (t == 0 && layer == 0 && h == 0 && p.err) atomicOr(p.err, kErrBadInput);
        return;
    }
    if (!(flags & 2)) return;   // every accepted row is already in place
    const int r16 = p.row_bytes / 16;
    const int64_t head_off = (((int64_t)b * p.Hkv + h) * p.cap + P) * p.row_bytes;
    uint8_t* kbase = static_cast<uint8_t*>(p.K[layer]) + head_off;
    uint8_t* vbase = static_cast<uint8_t*>(p.V[layer]) + head_off;
    const int total = n * r16;
    uint4* sk = staged;
    uint4* sv = staged + (p.n_q - 1) * r16;
    for (int x = t; x < total; x += kCommitThreads) {
        const int k = x / r16, c = x - k * r16;
        const int64_t src = (int64_t)s_src[k] * p.row_bytes;
        sk[x] = reinterpret_cast<const uint4*>(kbase + src)[c];
        sv[x] = reinterpret_cast<const uint4*>(vbase + src)[c];
    }
    __syncthreads();
    for (int x = t; x < total; x += kCommitThreads) {
        const int k = x / r16, c = x - k * r16;
        const int64_t dst = (int64_t)(1 + k) * p.row_bytes;
        reinterpret_cast<uint4*>(kbase + dst)[c] = sk[x];
        reinterpret_cast<uint4*>(vbase + dst)[c] = sv[x];
    }
}

__global__ void kv_advance_kernel(int32_t* prefix_len, const int32_t* n_acc, int B, int n_q,
                                  int64_t cap, unsigned int* err) {
    griddep_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int n = n_acc[b];
    const int64_t P = prefix_len[b];
    if (n < 0 || n > n_q - 1 || P < 0 || P + n_q > cap) {
        if (err) atomicOr(err, kErrBadInput);
        return;
    }
    prefix_len[b] = (int32_t)(P + 1 + n);
}

}  // namespace

cudaError_t launch_kv_commit(const CommitParams& p, cudaStream_t st) {
    const size_t smem = (size_t)2 * (p.n_q - 1) * p.row_bytes;
    cudaError_t e = cudaFuncSetAttribute(kv_commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(smem > 0 ? smem : 16));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.Hkv, p.layers, 1);
    cfg.blockDim = dim3(kCommitThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_commit_kernel, p);
}

cudaError_t launch_kv_advance(int32_t* prefix_len, const int32_t* n_acc, int B, int n_q,
                              int64_t cap, unsigned int* err, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((B + 127) / 128, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_advance_kernel, prefix_len, n_acc, B, n_q, cap, err);
}

}  // namespace rapid
